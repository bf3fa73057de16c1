// tv_tree_accept: longest accepted root-to-node path of the draft tree.
//
// Greedy (T = 0): a non-root node hits when its drafted token equals the
// target's argmax at its parent (the argmax rule of "SGLang EAGLE-2
// Speculative Decoding", section 2, applied to the target); the deepest node
// whose whole root path hits is accepted, and the target's argmax there is
// the bonus token (study note "EAGLE", case 1: k hits emit k+1 tokens).
//
// Sampling (T > 0): rejection sampling with residual resampling
// (troisinh.com "Why it works"; study note case 3).  At node n with
// p = softmax(target[n]/T) and q = softmax(draft[n]/T) the children are tried
// in ascending index: accept iff u*q(x) < p(x); after a rejection p becomes
// max(0, p - q) normalised.  When every child is rejected (or n is a leaf)
// the bonus is drawn from the current p by inverse CDF.
//
// Design: one thread-block cluster of CL CTAs per request: 8, or 16 or 12 for
// a sampling batch small enough that all its clusters of that size are
// resident at once (the residual passes then cover a smaller slice per CTA),
// or 4 for a greedy batch whose 8-CTA clusters would not all be resident.  CTA r owns the
// vocabulary slice [r*chunk, (r+1)*chunk).  Rows are read from HBM only for
// the nodes the walk visits; in sampling mode the visited node's p and q
// slices stay in shared memory for the residual passes and the inverse CDF.
// Cluster-wide reductions go through distributed shared memory and are
// combined in rank order, so every CTA takes identical decisions (uniform
// control flow across the cluster).
#include <cooperative_groups.h>
#include <cfloat>
#include <climits>
#include "tv_common.cuh"

namespace cg = cooperative_groups;

namespace tv {

constexpr int kCL = 8;             // CTAs per request when 16 would not all be resident
constexpr int kMinCL = 4;          // CTAs per request for large greedy batches (all clusters resident)
constexpr int kMidCL = 12;         // CTAs per request for sampling batches that fit as 12-CTA clusters
constexpr int kMaxCL = 16;         // CTAs per request for small sampling batches (non-portable cluster size)
constexpr int kAccThreads = 512;
constexpr int kAccWarps = kAccThreads / 32;
constexpr int kMaxChunk = 26624;  // floats per CTA and array (sampling keeps two arrays)

struct AcceptParams {
  const float* target;
  const float* draft;
  const int32_t* tokens;
  const int32_t* parents;
  const int32_t* n_nodes;
  const float* u_accept;
  const float* u_sample;
  int n_max, V, chunk;
  float k2;          // log2(e) / T   (sampling)
  int sampling;
  int wor;           // siblings drafted without replacement: q renormalised without each rejected token
  int32_t* accept_len;
  int32_t* path_nodes;
  int32_t* out_tokens;
  int32_t* status;
};

// Double-float numbers: value = hi + lo with |lo| <= ulp(hi) / 2 (about 48
// significant bits).  The sampling walk accumulates its sums, scans and
// thresholds in this form on the fp32 pipe; fp64 throughput is far too low on
// this GPU for a per-thread hot loop.  Sums use Knuth's TwoSum, products an
// fma-based TwoProduct (Dekker/Knuth error-free transformations).
struct Df {
  float hi, lo;
};
__device__ __forceinline__ Df df_norm(float s, float e) {
  const float hi = s + e;
  return {hi, e - (hi - s)};
}
__device__ __forceinline__ Df df_add(Df a, Df b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  const float e = (a.hi - (s - bb)) + (b.hi - bb) + (a.lo + b.lo);
  return df_norm(s, e);
}
__device__ __forceinline__ Df df_add1(Df a, float b) {
  const float s = a.hi + b;
  const float bb = s - a.hi;
  const float e = (a.hi - (s - bb)) + (b - bb) + a.lo;
  return df_norm(s, e);
}
__device__ __forceinline__ Df df_mul1(Df a, float u) {
  const float p = a.hi * u;
  const float e = fmaf(a.lo, u, fmaf(a.hi, u, -p));
  return df_norm(p, e);
}
__device__ __forceinline__ bool df_gt(Df a, Df b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }
__device__ __forceinline__ bool df_pos(Df a) { return a.hi > 0.f; }
__device__ __forceinline__ Df df_shfl_xor(Df a, int o) {
  return {__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ Df df_shfl_up(Df a, int o) {
  return {__shfl_up_sync(0xffffffffu, a.hi, o), __shfl_up_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ Df df_shfl(Df a, int src) {
  return {__shfl_sync(0xffffffffu, a.hi, src), __shfl_sync(0xffffffffu, a.lo, src)};
}

struct __align__(16) ClSlot {
  Df d[2];
  float f[2];
  int i[2];
};

struct AccShared {
  int par[kMaxNodes];
  int tok[kMaxNodes];
  int kid_off[kMaxNodes + 1];
  int kids[kMaxNodes];
  int am[kMaxNodes];
  int front[kMaxNodes];
  int nxt[kMaxNodes];
  int path[kMaxNodes];
  float wf[kAccWarps];
  int wi[kAccWarps];
  Df wd[kAccWarps][2];
  Df thr_excl[kAccThreads];  // exclusive scan of per-thread sums (inverse CDF)
  ClSlot slot[2];
  ClSlot gath[kMaxCL];  // this exchange's slots of every CTA, copied in (rank order)
  float ua[kMaxNodes];
  float bf;
  int bi;
  Df bd[2];
  float cf[2];
  uint64_t load_bar;
  int timed_out;
  int bad;
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

// Two block maxima at once; result in sh.cf (after a barrier).
__device__ void block_max2(float u, float v, AccShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    u = fmaxf(u, __shfl_xor_sync(0xffffffffu, u, o));
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  }
  if (lane == 0) {
    sh.wf[warp] = u;
    sh.wd[warp][0].hi = v;
  }
  __syncthreads();
  if (warp == 0) {
    u = lane < kAccWarps ? sh.wf[lane] : -FLT_MAX;
    v = lane < kAccWarps ? sh.wd[lane][0].hi : -FLT_MAX;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      u = fmaxf(u, __shfl_xor_sync(0xffffffffu, u, o));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    }
    if (lane == 0) {
      sh.cf[0] = u;
      sh.cf[1] = v;
    }
  }
  __syncthreads();
}

// Two double-float sums over the block; result in sh.bd (after a barrier).
__device__ void block_sum2(Df a, Df b, AccShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    a = df_add(a, df_shfl_xor(a, o));
    b = df_add(b, df_shfl_xor(b, o));
  }
  if (lane == 0) {
    sh.wd[warp][0] = a;
    sh.wd[warp][1] = b;
  }
  __syncthreads();
  if (warp == 0) {
    Df x = lane < kAccWarps ? sh.wd[lane][0] : Df{0.f, 0.f};
    Df y = lane < kAccWarps ? sh.wd[lane][1] : Df{0.f, 0.f};
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      x = df_add(x, df_shfl_xor(x, o));
      y = df_add(y, df_shfl_xor(y, o));
    }
    if (lane == 0) {
      sh.bd[0] = x;
      sh.bd[1] = y;
    }
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

// One pass over this CTA's slices after a rejected child: apply the deferred
// residual update of the previous rejection (pending), and sum the new
// residual max(0, w / Sw - q / Sq) into z.  Without replacement (kWor) the
// previously rejected token's draft weight is zeroed once the deferred update
// has used it, and the draft weights left after removing this child's token
// are summed into zq.  Products and differences are rounded one by one so
// every pass and every CTA agrees.
template <bool kWor>
__device__ __forceinline__ void residual_pass(float* wt, float* wq, int len, bool pending, float pend_isw,
                                              float pend_isq, int pend_zero, float cur_isw, float cur_isq,
                                              int xk_off, Df& z, Df& zq) {
  for (int j0 = threadIdx.x; j0 < len; j0 += 4 * kAccThreads) {
    float g = 0.f, gq = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u * kAccThreads;
      if (j < len) {
        float w = wt[j];
        float qw = wq[j];
        if (kWor) {
          if (pending) {
            w = fmaxf(0.f, __fsub_rn(__fmul_rn(w, pend_isw), __fmul_rn(qw, pend_isq)));
            wt[j] = w;
          }
          if (j == pend_zero) {
            qw = 0.f;
            wq[j] = 0.f;
          }
          g += fmaxf(0.f, __fsub_rn(__fmul_rn(w, cur_isw), __fmul_rn(qw, cur_isq)));
          if (j != xk_off) gq += qw;
        } else {  // the draft and its normaliser never change
          const float qq = __fmul_rn(qw, cur_isq);
          if (pending) {
            w = fmaxf(0.f, __fsub_rn(__fmul_rn(w, pend_isw), qq));
            wt[j] = w;
          }
          g += fmaxf(0.f, __fsub_rn(__fmul_rn(w, cur_isw), qq));
        }
      }
    }
    z = df_add1(z, g);
    if (kWor) zq = df_add1(zq, gq);
  }
}

// ---------------------------------------------------------------- the kernel
template <int CL>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(kAccThreads, 1)
    tree_accept_kernel(const AcceptParams p) {
  extern __shared__ __align__(16) float dyn[];
  __shared__ AccShared sh;
  ClusterEx<CL> ex;
  const int rank = (int)ex.cl.block_rank();
  const int b = blockIdx.x / CL;
  const int tid = threadIdx.x;
  const int n_max = p.n_max, V = p.V;
  const int lo = min(V, rank * p.chunk);
  const int hi = min(V, lo + p.chunk);
  const int len = hi - lo;
  float* wt = dyn;             // sampling: current target weights of this slice
  float* wq = dyn + p.chunk;   // sampling: draft weights of this slice

  // Everything up to the outputs reads only inputs (tree, tokens, logits,
  // uniforms) and writes nothing global, so it runs while the previous kernel
  // finishes; status, which that kernel may write, is read and written after the
  // wait before the outputs.
  // ---- tree setup and validation (every CTA redundantly, identical results):
  // one node per thread, then thread 0 builds the child lists from shared memory
  const int N = p.n_nodes[b];
  const bool n_ok = N >= 1 && N <= n_max;
  bool sbad = false, tbad = false;
  if (n_ok && tid < N) {
    const int pi = p.parents[(int64_t)b * n_max + tid];
    const int ti = p.tokens[(int64_t)b * n_max + tid];
    sh.par[tid] = pi;
    sh.tok[tid] = ti;
    sbad = tid == 0 ? pi != -1 : (pi < 0 || pi >= tid);
    tbad = tid >= 1 && (ti < 0 || ti >= V);
  }
  if (tid == 0) {
    mbar_init(&sh.load_bar, 1);
    fence_barrier_init();
    sh.timed_out = 0;
  }
  const bool any_s = __syncthreads_or(sbad) != 0;
  const bool any_t = __syncthreads_or(tbad) != 0;
  const int bad = (!n_ok || any_s) ? TV_DEV_BAD_TREE : (any_t ? TV_DEV_BAD_TOKEN : 0);
  if (bad == 0 && tid < kMaxNodes) {  // warps 0 and 1, whole
    // children of node tid, then the exclusive scan of the counts over the nodes
    int cnt = 0;
    if (tid < N)
      for (int j = 1; j < N; ++j) cnt += sh.par[j] == tid;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if ((tid & 31) >= o) incl += y;
    }
    if (tid == 31) sh.cnt = incl;  // warp 0's total
    if (tid < N) {
      sh.kid_off[tid] = incl - cnt;
      if (p.sampling) sh.ua[tid] = p.u_accept[(int64_t)b * n_max + tid];
    }
  }
  if (tid == 0) sh.bad = bad;
  __syncthreads();
  if (bad == 0 && tid < N) {
    if (tid >= 32) sh.kid_off[tid] += sh.cnt;
    if (tid == N - 1) sh.kid_off[N] = N - 1;  // every non-root node is somebody's child
  }
  __syncthreads();
  if (bad == 0 && tid >= 1 && tid < N) {
    // ascending child index within each parent's list
    const int pj = sh.par[tid];
    int before = 0;
    for (int k = 1; k < tid; ++k) before += sh.par[k] == pj;
    sh.kids[sh.kid_off[pj] + before] = tid;
  }
  __syncthreads();
  int best = 0;
  int bonus = -1;
  if (sh.bad == 0) {  // uniform across the cluster: every CTA computed the same flag
    const bool vec4 = (V & 3) == 0;

    if (!p.sampling) {
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
            s->f[0] = sh.bf;
            s->i[0] = sh.bi;
          }
          ex.exchange(sh);
          float gv = -FLT_MAX;
          int gi = INT_MAX;
          for (int r = 0; r < CL; ++r) {
            const ClSlot* s = ex.got(sh, r);
            argmax_take(gv, gi, s->f[0], s->i[0]);
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
            for (int k = sh.kid_off[node]; k < sh.kid_off[node + 1]; ++k) {
              const int c = sh.kids[k];
              if (sh.tok[c] == sh.am[node]) {
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
    } else {
      // ================================================ sampling: walk from the root
      int node = 0;
      uint32_t load_phase = 0;
      for (;;) {
        // this thread's accesses to the slices precede the next copy into them (the
        // last exchange was a barrier; no CTA reads another CTA's slices)
        fence_proxy_async_smem();
        const float* trow = p.target + ((int64_t)b * n_max + node) * V + lo;
        const float* drow = p.draft + ((int64_t)b * n_max + node) * V + lo;
        if (vec4) {
          // 16-byte aligned slices: two bulk copies into shared memory
          if (tid == 0) {
            mbar_arrive_expect_tx(&sh.load_bar, 8u * (uint32_t)len);
            if (len > 0) {
              bulk_g2s(wt, trow, 4u * (uint32_t)len, &sh.load_bar);
              bulk_g2s(wq, drow, 4u * (uint32_t)len, &sh.load_bar);
            }
          }
          if (!mbar_wait(&sh.load_bar, load_phase, &sh.timed_out)) sh.timed_out = 1;
          load_phase ^= 1u;
        } else {
          for (int j = tid; j < len; j += kAccThreads) {
            wt[j] = __ldg(trow + j);
            wq[j] = __ldg(drow + j);
          }
          __syncthreads();
        }
        float mt = -FLT_MAX, mq = -FLT_MAX;
        for (int j = tid; j < len; j += kAccThreads) {
          mt = fmaxf(mt, wt[j]);
          mq = fmaxf(mq, wq[j]);
        }
        block_max2(mt, mq, sh);
        if (tid == 0) {
          ClSlot* s = ex.publish(sh);
          s->f[0] = sh.cf[0];
          s->f[1] = sh.cf[1];
        }
        ex.exchange(sh);
        float Mt = -FLT_MAX, Mq = -FLT_MAX;
        for (int r = 0; r < CL; ++r) {
          const ClSlot* s = ex.got(sh, r);
          Mt = fmaxf(Mt, s->f[0]);
          Mq = fmaxf(Mq, s->f[1]);
        }
        ex.flip();
        // exponentiate in place: w = 2^((z - max) * log2(e)/T); sums in double-float
        // (four terms in fp32, then into the double-float sum)
        Df st{0.f, 0.f}, sq{0.f, 0.f};
        for (int j0 = tid; j0 < len; j0 += 4 * kAccThreads) {
          float gt = 0.f, gq = 0.f;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int j = j0 + u * kAccThreads;
            if (j < len) {
              const float et = exp2f((wt[j] - Mt) * p.k2);
              const float eq = exp2f((wq[j] - Mq) * p.k2);
              wt[j] = et;
              wq[j] = eq;
              gt += et;
              gq += eq;
            }
          }
          st = df_add1(st, gt);
          sq = df_add1(sq, gq);
        }
        block_sum2(st, sq, sh);
        const int k_beg = sh.kid_off[node], k_end = sh.kid_off[node + 1];
        int f_owner = 0, f_off = 0;
        if (k_beg < k_end) {
          const int x = sh.tok[sh.kids[k_beg]];
          f_owner = x / p.chunk;
          f_off = x - f_owner * p.chunk;
        }
        if (tid == 0) {
          ClSlot* s = ex.publish(sh);
          s->d[0] = sh.bd[0];
          s->d[1] = sh.bd[1];
          if (k_beg < k_end && rank == f_owner) {
            s->f[0] = wt[f_off];
            s->f[1] = wq[f_off];
          }
        }
        ex.exchange(sh);
        Df St{0.f, 0.f}, Sq{0.f, 0.f};
        for (int r = 0; r < CL; ++r) {  // rank order: identical in every CTA
          const ClSlot* s = ex.got(sh, r);
          St = df_add(St, s->d[0]);
          Sq = df_add(Sq, s->d[1]);
        }
        float pv0 = 0.f, qv0 = 0.f;
        if (k_beg < k_end) {
          pv0 = ex.got(sh, f_owner)->f[0];
          qv0 = ex.got(sh, f_owner)->f[1];
        }
        ex.flip();
        float Sw = St.hi;   // normaliser of the current target weights wt
        float SqF = Sq.hi;  // normaliser of the current draft weights wq
        // the tested child's numerators: the owner CTA published them in the exchange
        // (no CTA reads another CTA's slices during the walk)
        float pv = pv0, qv = qv0;
        // a residual step whose slice update is deferred to the next pass:
        // wt = max(0, wt * pend_isw - wq * pend_isq), its normaliser already in Sw
        bool pending = false;
        float pend_isw = 0.f, pend_isq = 0.f;
        // without replacement: the rejected token whose draft weight is zeroed in the
        // next pass, after that pass's deferred update has used it (slice offset, or -1)
        int pend_zero = -1;
        int accepted = -1;
        for (int k = k_beg; k < k_end; ++k) {
          const int c = sh.kids[k];
          const float u = sh.ua[c];
          if (u * (SqF > 0.f ? qv / SqF : 0.f) < pv / Sw) {
            accepted = c;
            break;
          }
          // rejected: the residual max(0, p - q), normalised (p kept if it sums to 0);
          // without replacement also q without the rejected token, renormalised.  One
          // pass applies the deferred update and sums the new residual (and the
          // remaining draft weights); products and differences are rounded one by one
          // so every pass agrees.
          const float cur_isw = 1.f / Sw;
          const float cur_isq = SqF > 0.f ? 1.f / SqF : 0.f;
          const int xk = sh.tok[c];
          const int xk_off = (p.wor && xk >= lo && xk < hi) ? xk - lo : -1;
          Df z{0.f, 0.f}, zq{0.f, 0.f};
          if (p.wor)
            residual_pass<true>(wt, wq, len, pending, pend_isw, pend_isq, pend_zero, cur_isw, cur_isq, xk_off, z, zq);
          else
            residual_pass<false>(wt, wq, len, pending, pend_isw, pend_isq, pend_zero, cur_isw, cur_isq, xk_off, z, zq);
          block_sum2(z, zq, sh);
          const bool more = k + 1 < k_end;
          int nx_owner = 0, nx_off = 0, nx_tok = -1;
          if (more) {
            nx_tok = sh.tok[sh.kids[k + 1]];
            nx_owner = nx_tok / p.chunk;
            nx_off = nx_tok - nx_owner * p.chunk;
          }
          if (tid == 0) {
            ClSlot* s = ex.publish(sh);
            s->d[0] = sh.bd[0];
            s->d[1] = sh.bd[1];
            if (more && rank == nx_owner) {
              const float w = wt[nx_off];
              const float qw = wq[nx_off];
              s->f[0] = w;                                                   // p numerator if kept
              s->f[1] = (p.wor && nx_tok == xk) ? 0.f : qw;                  // next child's q numerator
              s->i[0] = __float_as_int(
                  fmaxf(0.f, __fsub_rn(__fmul_rn(w, cur_isw), __fmul_rn(qw, cur_isq))));  // residual numerator
            }
          }
          ex.exchange(sh);
          Df Z{0.f, 0.f}, Zq{0.f, 0.f};
          for (int r = 0; r < CL; ++r) {
            Z = df_add(Z, ex.got(sh, r)->d[0]);
            Zq = df_add(Zq, ex.got(sh, r)->d[1]);
          }
          float nw = 0.f, nq = 0.f, nr = 0.f;
          if (more) {
            const ClSlot* o = ex.got(sh, nx_owner);
            nw = o->f[0];
            nq = o->f[1];
            nr = __int_as_float(o->i[0]);
          }
          ex.flip();
          if (df_pos(Z)) {
            pending = true;
            pend_isw = cur_isw;
            pend_isq = cur_isq;
            Sw = Z.hi;
            pv = nr;
          } else {
            pending = false;
            pv = nw;
          }
          if (p.wor) {
            pend_zero = xk_off;
            SqF = Zq.hi;
          }
          qv = nq;
        }
        if (accepted >= 0) {
          node = accepted;
          continue;
        }
        if (pending) {  // the bonus draw reads the current p: apply the deferred update
          for (int j = tid; j < len; j += kAccThreads)
            wt[j] = fmaxf(0.f, __fsub_rn(__fmul_rn(wt[j], pend_isw), __fmul_rn(wq[j], pend_isq)));
          __syncthreads();
        }
        // ---- bonus token: inverse CDF of wt with u_sample[node] (double-float prefix sums)
        {
          const int per = (len + kAccThreads - 1) / kAccThreads;
          const int a0 = min(len, tid * per), a1 = min(len, a0 + per);
          // this thread's range sum, starting at an offset rotated by the lane so that
          // the 32 lanes hit 32 different banks (the ranges are `per` words apart)
          Df tsum{0.f, 0.f};
          {
            const int cnt = a1 - a0;
            int jj = cnt > 0 ? (tid & 31) % cnt : 0;
            for (int n = 0; n < cnt; ++n) {
              tsum = df_add1(tsum, wt[a0 + jj]);
              jj = (jj + 1 == cnt) ? 0 : jj + 1;
            }
          }
          // exclusive scan over the block's threads
          const int lane = tid & 31, warp = tid >> 5;
          Df incl = tsum;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const Df y = df_shfl_up(incl, o);
            if (lane >= o) incl = df_add(incl, y);
          }
          Df prev = df_shfl_up(incl, 1);
          if (lane == 0) prev = Df{0.f, 0.f};
          if (lane == 31) sh.wd[warp][0] = incl;
          __syncthreads();
          if (tid == 0) {
            Df run{0.f, 0.f};
            for (int w = 0; w < kAccWarps; ++w) {
              const Df t = sh.wd[w][0];
              sh.wd[w][1] = run;
              run = df_add(run, t);
            }
            sh.bd[0] = run;
          }
          __syncthreads();
          sh.thr_excl[tid] = df_add(sh.wd[warp][1], prev);
          const Df s_r = sh.bd[0];
          if (tid == 0) {
            ClSlot* s = ex.publish(sh);
            s->d[0] = s_r;
          }
          ex.exchange(sh);
          Df pre[CL], srk[CL];
          Df S{0.f, 0.f};
          for (int r = 0; r < CL; ++r) {
            pre[r] = S;
            srk[r] = ex.got(sh, r)->d[0];
            S = df_add(S, srk[r]);
          }
          ex.flip();
          const Df t = df_mul1(S, p.u_sample[(int64_t)b * n_max + node]);
          int rstar = -1, rlast = -1;
          for (int r = 0; r < CL; ++r) {
            if (df_pos(srk[r])) rlast = r;
            if (rstar < 0 && df_gt(df_add(pre[r], srk[r]), t)) rstar = r;
          }
          const bool fallback_rank = rstar < 0;
          if (fallback_rank) rstar = rlast;
          int found = -1;
          if (rank == rstar) {
            // thread whose range crosses t (or the last non-empty one on fallback)
            const Df base = df_add(pre[rank], sh.thr_excl[tid]);
            const bool nonempty = tsum.hi > 0.f;
            const bool crosses = !fallback_rank && nonempty && df_gt(df_add(base, tsum), t) && !df_gt(base, t);
            if (tid == 0) {
              sh.bi = INT_MAX;
              sh.wi[0] = -1;
            }
            __syncthreads();
            if (crosses) atomicMin(&sh.bi, tid);
            if (nonempty) atomicMax(&sh.wi[0], tid);
            __syncthreads();
            int kstar = sh.bi;
            const bool fb = (kstar == INT_MAX);
            if (fb) kstar = sh.wi[0];
            if (tid == kstar) {
              Df acc = base;
              int j_found = -1, j_last = -1;
              for (int j = a0; j < a1; ++j) {
                if (wt[j] > 0.f) j_last = j;
                acc = df_add1(acc, wt[j]);
                if (!fb && j_found < 0 && df_gt(acc, t) && wt[j] > 0.f) j_found = j;
              }
              sh.wi[1] = lo + (j_found >= 0 ? j_found : j_last);
            }
            __syncthreads();
            found = sh.wi[1];
          }
          if (tid == 0) {
            ClSlot* s = ex.publish(sh);
            s->i[0] = found;
          }
          ex.exchange(sh);
          int tokv = -1;
          for (int r = 0; r < CL; ++r) tokv = max(tokv, ex.got(sh, r)->i[0]);
          ex.flip();
          bonus = tokv;
        }
        best = node;
        break;
      }
    }
  }  // sh.bad == 0

  // ---- outputs (rank 0), after the previous kernel: a request flagged on entry,
  // or with an invalid tree, gets an empty path
  griddep_wait();
  const int st_in = p.status[b];
  const int bad_out = st_in != 0 ? -1 : sh.bad;
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
    if (sh.timed_out) atomicOr(p.status + b, TV_DEV_TIMEOUT);
    int len_path = 0;
    for (int j = best; j != 0; j = sh.par[j]) sh.path[len_path++] = j;
    // sh.path holds best .. first child; emit root-first
    int32_t* pn = p.path_nodes + (int64_t)b * n_max;
    int32_t* ot = p.out_tokens + (int64_t)b * (n_max + 1);
    pn[0] = 0;
    for (int k = 1; k <= len_path; ++k) {
      const int nd = sh.path[len_path - k];
      pn[k] = nd;
      ot[k - 1] = sh.tok[nd];
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
// CTAs per request: for sampling, the largest of 16 and 12 whose clusters of
// the whole batch can be resident at once (non-portable sizes allowed, at
// least B such clusters active), else 8.  0 when a CUDA call fails.
template <int CL>
int active_clusters(int dev) {
  static int known[64] = {};  // per device: clusters of CL that fit at once, plus 1 (0 = not yet known)
  static unsigned long long ctx_of[64] = {};  // the context the attributes were set in
  unsigned long long ctx = 0;
  if (tv::current_context_id(&ctx) != cudaSuccess) return -1;
  if (known[dev] == 0 || ctx == 0 || ctx_of[dev] != ctx) {
    const void* f = (const void*)tv::tree_accept_kernel<CL>;
    if (cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) return -1;
    if (tv::ensure_smem_attr(f, 2ull * tv::kMaxChunk * sizeof(float)) != cudaSuccess) return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL);
    cfg.blockDim = dim3(tv::kAccThreads);
    cfg.dynamicSmemBytes = 2ull * tv::kMaxChunk * sizeof(float);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tv::tree_accept_kernel<CL>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    known[dev] = n + 1;
    if (tv::current_context_id(&ctx_of[dev]) != cudaSuccess) ctx_of[dev] = 0;
  }
  return known[dev] - 1;
}

int accept_cluster_size(bool sampling, int B) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int sms = tv::current_sm_count();
  if (!sampling) {
    // greedy level walk: 8 CTAs per request unless the batch's 8-CTA clusters
    // cannot all be resident at once, then 4
    if ((int64_t)B * tv::kCL <= sms) return tv::kCL;
    const int n8 = active_clusters<tv::kCL>(dev);
    if (n8 < 0) return 0;
    return n8 >= B ? tv::kCL : tv::kMinCL;
  }
  if ((int64_t)B * tv::kMaxCL <= sms) {
    const int n = active_clusters<tv::kMaxCL>(dev);
    if (n < 0) return 0;
    if (n >= B) return tv::kMaxCL;
  }
  if ((int64_t)B * tv::kMidCL <= sms) {
    const int n = active_clusters<tv::kMidCL>(dev);
    if (n < 0) return 0;
    if (n >= B) return tv::kMidCL;
  }
  return tv::kCL;
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
  const int cl = accept_cluster_size(sampling, B);
  TV_REQUIRE(cl > 0, TV_ERR_CUDA, "tv_tree_accept: cluster attribute query failed");
  const int per = (V + cl - 1) / cl;
  const int chunk = (per + 3) & ~3;
  TV_REQUIRE(!sampling || chunk <= tv::kMaxChunk, TV_ERR_UNSUPPORTED,
             "tv_tree_accept: V = %d too large for on-chip sampling (max %d)", V, tv::kMaxChunk * cl);
  if (!sampling && onepass_eligible(B, n_max, V)) {
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
  TV_REQUIRE((int64_t)B * cl < (1ll << 31), TV_ERR_UNSUPPORTED, "tv_tree_accept: B too large");
  tv::AcceptParams p;
  p.target = target_logits;
  p.draft = draft_logits;
  p.tokens = tokens;
  p.parents = parents;
  p.n_nodes = n_nodes;
  p.u_accept = u_accept;
  p.u_sample = u_sample;
  p.n_max = n_max;
  p.V = V;
  p.chunk = chunk;
  p.k2 = sampling ? (float)(1.4426950408889634 / (double)temperature) : 0.f;
  p.sampling = sampling ? 1 : 0;
  p.wor = (flags & TV_ACCEPT_SIBLINGS_WITHOUT_REPLACEMENT) ? 1 : 0;
  p.accept_len = accept_len;
  p.path_nodes = path_nodes;
  p.out_tokens = out_tokens;
  p.status = status;
  const size_t smem = sampling ? 2ull * chunk * sizeof(float) : 0;
  if (cl == tv::kMaxCL) {
    TV_CUDA_CHECK(tv::ensure_smem_attr((const void*)tv::tree_accept_kernel<tv::kMaxCL>,
                                       2ull * tv::kMaxChunk * sizeof(float)));
    TV_CUDA_CHECK(tv::launch_pdl(tv::tree_accept_kernel<tv::kMaxCL>, dim3(B * cl), dim3(tv::kAccThreads), smem,
                                 tv::as_stream(stream), p));
  } else if (cl == tv::kMinCL) {
    TV_CUDA_CHECK(tv::ensure_smem_attr((const void*)tv::tree_accept_kernel<tv::kMinCL>,
                                       2ull * tv::kMaxChunk * sizeof(float)));
    TV_CUDA_CHECK(tv::launch_pdl(tv::tree_accept_kernel<tv::kMinCL>, dim3(B * cl), dim3(tv::kAccThreads), smem,
                                 tv::as_stream(stream), p));
  } else if (cl == tv::kMidCL) {
    TV_CUDA_CHECK(tv::ensure_smem_attr((const void*)tv::tree_accept_kernel<tv::kMidCL>,
                                       2ull * tv::kMaxChunk * sizeof(float)));
    TV_CUDA_CHECK(tv::launch_pdl(tv::tree_accept_kernel<tv::kMidCL>, dim3(B * cl), dim3(tv::kAccThreads), smem,
                                 tv::as_stream(stream), p));
  } else {
    TV_CUDA_CHECK(tv::ensure_smem_attr((const void*)tv::tree_accept_kernel<tv::kCL>,
                                       2ull * tv::kMaxChunk * sizeof(float)));
    TV_CUDA_CHECK(tv::launch_pdl(tv::tree_accept_kernel<tv::kCL>, dim3(B * cl), dim3(tv::kAccThreads), smem,
                                 tv::as_stream(stream), p));
  }
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
}
