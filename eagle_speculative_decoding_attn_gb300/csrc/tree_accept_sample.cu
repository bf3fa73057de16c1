// tv_tree_accept, sampling (T > 0): rejection sampling with residual
// resampling over the draft tree (troisinh.com "Why it works"; study note
// "EAGLE", case 3).  At node n with p = softmax(target[n]/T) and
// q = softmax(draft[n]/T) the children are tried in ascending index: accept iff
// u*q(x) < p(x); after a rejection p becomes max(0, p - q) normalised (kept
// when that is all zero).  When every child is rejected (or n is a leaf) the
// bonus token is drawn from the current p by inverse CDF.
//
// Closed form of the residual.  With unnormalised weights e_t = exp(z_t/T),
// e_q = exp(z_q/T) and S_q = sum e_q, the residual after k rejections at a node
// is N_k = max(0, e_t - c_k e_q) for a scalar c_k: c_0 = 0 and
// c_{k+1} = c_k + R_k / S_q with R_k = sum N_k, because
// max(0, max(0, y) - d) = max(0, y - d) for d >= 0.  A rejection therefore
// costs one fused multiply-add, a max and an add per vocabulary entry, and the
// logits never change after they are exponentiated.  Without replacement the
// draft also loses the rejected token x (q(x) <- 0, renormalised); x then keeps
// the residual weight it has at that step, which the kernel stores in its e_t
// slot with e_q(x) = 0, so the same closed form covers the later steps.
//
// Design.  One thread-block cluster of CL CTAs (CL <= 16, set at launch) per
// request; CTA r holds vocabulary entries [r*chunk, (r+1)*chunk), chunk =
// 512 * EPT, and thread t of it the EPT consecutive entries from
// r*chunk + t*EPT, target and draft, in registers.  Rows are read from HBM once
// per visited node.  Each CTA exponentiates against its own maxima; the
// cluster-wide sums weight CTA r's partials by alpha_r = 2^((m_r - M)*log2(e)/T).
// Cluster reductions do not use cluster barriers: every warp pushes its
// double-float partial into every CTA's shared memory with st.async, completing
// bytes on the receiver's mbarrier, and every warp of every CTA combines the
// 16*CL partials in the same fixed order, so all CTAs take identical decisions.
#include <cfloat>
#include <climits>
#include "tv_common.cuh"
#include "accept_common.cuh"

namespace tv {

namespace {

constexpr int kSmpThreads = 512;
constexpr int kSmpWarps = kSmpThreads / 32;
constexpr int kSmpMaxCL = 16;

struct SampleParams {
  const float* target;
  const float* draft;
  const int32_t* tokens;
  const int32_t* parents;
  const int32_t* n_nodes;
  const float* u_accept;
  const float* u_sample;
  int n_max, V, cl, chunk;
  float k2;  // log2(e) / T
  int32_t* accept_len;
  int32_t* path_nodes;
  int32_t* out_tokens;
  int32_t* status;
};

// ---------------------------------------------------------------- double-float
// value = hi + lo.  Sums of non-negative terms use Fast2Sum on the larger and
// the smaller high part (exact error term) and leave the low part
// unnormalised until the result is compared; products use an fma-based
// TwoProduct (Dekker/Knuth error-free transformations).  About 48 significant
// bits on the fp32 pipe.
struct Df {
  float hi, lo;
};
__device__ __forceinline__ Df dfp_add(Df a, Df b) {  // a, b >= 0
  const float x = fmaxf(a.hi, b.hi), y = fminf(a.hi, b.hi);
  const float s = x + y;
  const float e = y - (s - x);
  return {s, e + (a.lo + b.lo)};
}
__device__ __forceinline__ Df df_norm(Df a) {
  const float hi = a.hi + a.lo;
  return {hi, a.lo - (hi - a.hi)};
}
__device__ __forceinline__ Df df_mul1(Df a, float u) {
  const float p = a.hi * u;
  const float e = fmaf(a.lo, u, fmaf(a.hi, u, -p));
  return {p, e};
}
// a - b for normalised a >= b >= 0 (TwoSum of the high parts)
__device__ __forceinline__ Df df_sub(Df a, Df b) {
  const float s = a.hi - b.hi;
  const float bb = s - a.hi;
  const float e = (a.hi - (s - bb)) - (b.hi + bb) + (a.lo - b.lo);
  return df_norm({s, e});
}
__device__ __forceinline__ bool df_gt(Df a, Df b) {  // both normalised
  return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo);
}
__device__ __forceinline__ Df df_shfl_xor(Df a, int o) {
  return {__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ Df df_shfl_up(Df a, int o) {
  return {__shfl_up_sync(0xffffffffu, a.hi, o), __shfl_up_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ Df df_shfl(Df a, int src) {
  return {__shfl_sync(0xffffffffu, a.hi, src), __shfl_sync(0xffffffffu, a.lo, src)};
}
// sum over the warp, the same value in every lane
__device__ __forceinline__ Df warp_sum(Df a) {
#pragma unroll
  for (int o = 16; o; o >>= 1) a = dfp_add(a, df_shfl_xor(a, o));
  return a;
}

// fp32 sum of a register array by pairs (error bound log2(N) ulps)
template <int N>
__device__ __forceinline__ float pair_sum(const float (&v)[N]) {
  float s[N];
#pragma unroll
  for (int i = 0; i < N; ++i) s[i] = v[i];
#pragma unroll
  for (int w = 1; w < N; w <<= 1)
#pragma unroll
    for (int i = 0; i + w < N; i += 2 * w) s[i] += s[i + w];
  return s[0];
}
template <int N>
__device__ __forceinline__ float pair_max(const float (&v)[N]) {
  float s[N];
#pragma unroll
  for (int i = 0; i < N; ++i) s[i] = v[i];
#pragma unroll
  for (int w = 1; w < N; w <<= 1)
#pragma unroll
    for (int i = 0; i + w < N; i += 2 * w) s[i] = fmaxf(s[i], s[i + w]);
  return s[0];
}
// register element e of v (e uniform or not; no local-memory indexing)
template <int N>
__device__ __forceinline__ float reg_at(const float (&v)[N], int e) {
  float r = 0.f;
#pragma unroll
  for (int i = 0; i < N; ++i) r = i == e ? v[i] : r;
  return r;
}

// order-preserving float <-> int map (for integer max reductions)
__device__ __forceinline__ int f2ord(float f) {
  const int i = __float_as_int(f);
  return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float ord2f(int i) { return __int_as_float(i >= 0 ? i : i ^ 0x7fffffff); }

// ---------------------------------------------------------------- cluster pushes
__device__ __forceinline__ void st_async4(uint32_t raddr, float a, float b, float c, float d, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
               :: "r"(raddr), "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(__float_as_uint(c)),
                  "r"(__float_as_uint(d)), "r"(rbar)
               : "memory");
}
__device__ __forceinline__ void st_async2(uint32_t raddr, float a, float b, uint32_t rbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];"
               :: "r"(raddr), "r"(__float_as_uint(a)), "r"(__float_as_uint(b)), "r"(rbar)
               : "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

struct __align__(16) SmpShared {
  float4 recv[2][kSmpMaxCL][kSmpWarps];  // exchange x: (hi, lo, hi, lo) partials of every CTA's warps
  float2 recv_m[2][kSmpMaxCL];           // node visit v: every CTA's maxima (target, draft)
  float2 recv_kid[2][kMaxNodes];         // node visit v: the children's (e_t, e_q), by child position
  float2 kt[kSmpWarps][kMaxNodes];       // per warp: the children's current (e_t, e_q)
  float4 rk[kSmpWarps][kSmpMaxCL];       // per warp: per CTA (alpha, beta, beta / alpha, -) of the visit
  int2 wmax[2][kSmpWarps];
  uint64_t bar[2];
  uint64_t bar_cta;  // block barrier with a bounded wait (one arrival per warp)
  AccTree tr;
  int timed_out;
};

// This thread's EPT consecutive entries of a row, from token t0 (-inf past V).
template <int EPT>
__device__ __forceinline__ void load_slice(const float* row, int t0, int V, float (&v)[EPT]) {
  if ((V & 3) == 0) {  // rows 16-byte aligned, groups of four never straddle V
    const float4* r4 = reinterpret_cast<const float4*>(row + t0);
#pragma unroll
    for (int i = 0; i < EPT / 4; ++i) {
      float4 x = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      if (t0 + 4 * i < V) x = __ldcs(r4 + i);
      v[4 * i] = x.x;
      v[4 * i + 1] = x.y;
      v[4 * i + 2] = x.z;
      v[4 * i + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPT; ++i) v[i] = t0 + i < V ? __ldcs(row + t0 + i) : -INFINITY;
  }
}

template <int EPT, bool kWor>
__global__ void __launch_bounds__(kSmpThreads, 1) accept_sample_kernel(const SampleParams p) {
  __shared__ SmpShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int CL = p.cl;
  const int rank = (int)cluster_ctarank();
  const int b = blockIdx.x / CL;
  const int n_max = p.n_max, V = p.V;
  const int t0 = rank * p.chunk + tid * EPT;  // this thread's first token
  const float k2 = p.k2;

  // Everything up to the outputs reads only inputs (tree, tokens, logits,
  // uniforms) and writes nothing global, so it runs while the previous kernel
  // finishes.  The root's rows first: their loads overlap the tree setup.
  float a[EPT], q[EPT];
  load_slice<EPT>(p.target + (int64_t)b * n_max * V, t0, V, a);
  load_slice<EPT>(p.draft + (int64_t)b * n_max * V, t0, V, q);
  if (tid == 0) {
    mbar_init(&sh.bar[0], 1);
    mbar_init(&sh.bar[1], 1);
    mbar_init(&sh.bar_cta, kSmpWarps);
    fence_barrier_init();
    sh.timed_out = 0;
  }
  cluster_arrive();  // the barriers exist before any CTA pushes into them
  const int bad = acc_tree_setup(sh.tr, p.parents, p.tokens, p.u_accept, p.n_nodes, b, n_max, V);

  // remote addresses of this lane's target CTA (lanes 0..CL-1 push to CTA lane)
  const int tgt = lane < CL ? lane : 0;
  const uint32_t r_recv = mapa_shared(smem_u32(&sh.recv[0][0][0]), (uint32_t)tgt);
  const uint32_t r_recvm = mapa_shared(smem_u32(&sh.recv_m[0][0]), (uint32_t)tgt);
  const uint32_t r_bar = mapa_shared(smem_u32(&sh.bar[0]), (uint32_t)tgt);
  cluster_wait();

  int best = 0;
  int bonus_writer = 0;  // this thread writes the bonus token
  int bonus = -1;
  if (bad == 0) {  // uniform across the cluster
    int node = 0;
    int xb = 0;           // exchange buffer
    uint32_t phase = 0;   // bit x: parity of bar[x]
    uint32_t cta_phase = 0;
    volatile int* const aborted = &sh.timed_out;  // a wait gave up: leave the walk
    int vp = 0;           // node-visit buffer
    const int part_r = lane >> 1;  // bonus scan: lane's partials are CTA part_r, warps (lane & 1) * 8 + 0..7

    // wait for exchange xb, then flip the buffer
    auto exchange_wait = [&]() {
      if (!mbar_wait_cluster(&sh.bar[xb], (phase >> xb) & 1u, &sh.timed_out)) sh.timed_out = 1;
      phase ^= 1u << xb;
    };
    // the sum over every CTA's warp partials of exchange x (first or second
    // double-float of each slot); the same order in every warp and CTA
    auto gather_sum = [&](int x, bool second) {
      Df s{0.f, 0.f};
#pragma unroll
      for (int i = 0; i < kSmpWarps / 2; ++i) {
        const int slot = lane + 32 * i;  // CTA slot >> 4, warp slot & 15
        if ((slot >> 4) < CL) {
          const float4 v = sh.recv[x][slot >> 4][slot & 15];
          s = dfp_add(s, second ? Df{v.z, v.w} : Df{v.x, v.y});
        }
      }
      return df_norm(warp_sum(s));
    };

    for (;;) {
      // ---- node visit: this CTA's maxima (one block barrier)
      {
        const int it = __reduce_max_sync(0xffffffffu, f2ord(pair_max(a)));
        const int iq = __reduce_max_sync(0xffffffffu, f2ord(pair_max(q)));
        if (lane == 0) sh.wmax[vp][warp] = make_int2(it, iq);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.bar_cta);
      if (!mbar_wait(&sh.bar_cta, cta_phase, &sh.timed_out)) sh.timed_out = 1;
      cta_phase ^= 1u;
      if (*aborted) goto walk_end;
      float mt, mq;
      {
        const int2 w = sh.wmax[vp][lane & (kSmpWarps - 1)];
        mt = ord2f(__reduce_max_sync(0xffffffffu, w.x));
        mq = ord2f(__reduce_max_sync(0xffffffffu, w.y));
        if (mt == -INFINITY) mt = 0.f;  // an all-padding slice (weights 0)
        if (mq == -INFINITY) mq = 0.f;
      }
      // exponentiate against the CTA maxima; thread sums by pairs
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        a[e] = exp2f((a[e] - mt) * k2);
        q[e] = exp2f((q[e] - mq) * k2);
      }
      const Df wt = warp_sum({pair_sum(a), 0.f});
      const Df wq = warp_sum({pair_sum(q), 0.f});
      const int k_beg = sh.tr.kid_off[node], k_end = sh.tr.kid_off[node + 1];
      const int nk = k_end - k_beg;
      // publish: warp partials, CTA maxima (warp 0), children's weights (owners)
      if (tid == 0)  // every CTA's warp partials and maxima, one 8-byte push per child
        mbar_arrive_expect_tx(&sh.bar[xb], (uint32_t)(CL * (kSmpWarps * 16 + 8) + nk * 8));
      if (lane < CL) {
        st_async4(r_recv + (uint32_t)(((xb * kSmpMaxCL + rank) * kSmpWarps + warp) * 16), wt.hi, wt.lo, wq.hi,
                  wq.lo, r_bar + 8u * xb);
        if (warp == 0) st_async2(r_recvm + (uint32_t)((vp * kSmpMaxCL + rank) * 8), mt, mq, r_bar + 8u * xb);
      }
      for (int k = k_beg; k < k_end; ++k) {
        const int e = sh.tr.tok[sh.tr.kids[k]] - t0;
        if ((unsigned)e < (unsigned)EPT) {
          const float ax = reg_at(a, e), qx = reg_at(q, e);
          const uint32_t off = smem_u32(&sh.recv_kid[vp][k - k_beg]);
          const uint32_t bar = smem_u32(&sh.bar[xb]);
          for (int r = 0; r < CL; ++r) st_async2(mapa_shared(off, r), ax, qx, mapa_shared(bar, r));
        }
      }
      exchange_wait();
      if (*aborted) goto walk_end;
      // per-CTA weights alpha_r, beta_r against the global maxima
      {
        const float2 m = lane < CL ? sh.recv_m[vp][lane] : make_float2(-INFINITY, -INFINITY);
        const float Mt = ord2f(__reduce_max_sync(0xffffffffu, f2ord(m.x)));
        const float Mq = ord2f(__reduce_max_sync(0xffffffffu, f2ord(m.y)));
        if (lane < CL) {
          const float al = exp2f((m.x - Mt) * k2), be = exp2f((m.y - Mq) * k2);
          sh.rk[warp][lane] = make_float4(al, be, al > 0.f ? be / al : 0.f, 0.f);
        }
        for (int j = lane; j < nk; j += 32) sh.kt[warp][j] = sh.recv_kid[vp][j];
        __syncwarp();
      }
      Df R, Sq;  // current residual mass and draft mass, global scale
      {
        Df st{0.f, 0.f}, sq{0.f, 0.f};
#pragma unroll
        for (int i = 0; i < kSmpWarps / 2; ++i) {
          const int slot = lane + 32 * i;
          if ((slot >> 4) < CL) {
            const float4 v = sh.recv[xb][slot >> 4][slot & 15];
            const float4 f = sh.rk[warp][slot >> 4];
            st = dfp_add(st, df_mul1({v.x, v.y}, f.x));
            sq = dfp_add(sq, df_mul1({v.z, v.w}, f.y));
          }
        }
        R = df_norm(warp_sum(st));
        Sq = df_norm(warp_sum(sq));
      }
      const float4 mine = sh.rk[warp][rank];  // this CTA's (alpha, beta, beta / alpha)
      int src_x = xb;        // exchange holding the current distribution's partials
      bool src_scaled = false;  // ... already weighted by alpha (rejection passes are)
      int src_age = 0;       // exchanges since
      xb ^= 1;
      vp ^= 1;

      // ---- children in ascending index
      float cpr = 0.f;  // c_k
      int accepted = -1;
      for (int k = k_beg; k < k_end; ++k) {
        const int j = k - k_beg, c = sh.tr.kids[k], x = sh.tr.tok[c];
        const int o = x / p.chunk;
        const float4 fo = sh.rk[warp][o];
        const float2 v = sh.kt[warp][j];
        const float pn = fo.x * fmaxf(0.f, fmaf(-(cpr * fo.z), v.y, v.x));
        const float qn = fo.y * v.y;
        const float u = sh.tr.ua[c];
        if (u * (Sq.hi > 0.f ? qn / Sq.hi : 0.f) < pn / R.hi) {
          accepted = c;
          break;
        }
        // rejected: the next residual max(0, e_t - c' e_q), c' = c + R / S_q
        const float c_new = Sq.hi > 0.f ? cpr + R.hi / Sq.hi : cpr;
        const float g = c_new * mine.z;
        const int xe = x - t0;  // x's register in this thread, if in [0, EPT)
        float z[EPT], zq[EPT];
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
          z[e] = fmaxf(0.f, fmaf(-g, q[e], a[e]));
          if (kWor) zq[e] = e == xe ? 0.f : q[e];
        }
        Df dz = df_mul1(warp_sum({pair_sum(z), 0.f}), mine.x);
        Df dq{0.f, 0.f};
        if (kWor) dq = df_mul1(warp_sum({pair_sum(zq), 0.f}), mine.y);
        if (tid == 0) mbar_arrive_expect_tx(&sh.bar[xb], (uint32_t)(CL * kSmpWarps * 16));
        if (lane < CL)
          st_async4(r_recv + (uint32_t)(((xb * kSmpMaxCL + rank) * kSmpWarps + warp) * 16), dz.hi, dz.lo, dq.hi,
                    dq.lo, r_bar + 8u * xb);
        exchange_wait();
        if (*aborted) goto walk_end;
        const Df Z = gather_sum(xb, false);
        const bool kept = !(Z.hi > 0.f);  // an all-zero residual keeps p
        ++src_age;
        if (!kept) {
          src_x = xb;
          src_scaled = true;
          src_age = 0;
        }
        if (kWor) {
          // x leaves the draft and keeps its weight of the distribution now current
          const float c_eff = kept ? cpr : c_new;
          if ((unsigned)xe < (unsigned)EPT) {
            const float ge = c_eff * mine.z;
#pragma unroll
            for (int e = 0; e < EPT; ++e)
              if (e == xe) {
                a[e] = fmaxf(0.f, fmaf(-ge, q[e], a[e]));
                q[e] = 0.f;
              }
          }
          const float2 fz = make_float2(fmaxf(0.f, fmaf(-(c_eff * fo.z), v.y, v.x)), 0.f);
          for (int jj = lane; jj < nk; jj += 32)
            if (sh.tr.tok[sh.tr.kids[k_beg + jj]] == x) sh.kt[warp][jj] = fz;
          __syncwarp();
          Sq = gather_sum(xb, true);
        }
        if (!kept) {
          cpr = c_new;
          R = Z;
        }
        xb ^= 1;
      }
      if (accepted >= 0) {
        node = accepted;
        load_slice<EPT>(p.target + ((int64_t)b * n_max + node) * V, t0, V, a);
        load_slice<EPT>(p.draft + ((int64_t)b * n_max + node) * V, t0, V, q);
        continue;
      }

      // ---- bonus token: inverse CDF of the current distribution
      // N(v) = alpha_r * max(0, e_t - c e_q) in CTA r
      const float gcur = cpr * mine.z;
      float nv[EPT];
#pragma unroll
      for (int e = 0; e < EPT; ++e) nv[e] = fmaxf(0.f, fmaf(-gcur, q[e], a[e]));
      if (src_age > 1) {
        // the partials of the current distribution were overwritten (an all-zero
        // residual kept p twice in a row): publish them again
        const Df d = df_mul1(warp_sum({pair_sum(nv), 0.f}), mine.x);
        if (tid == 0) mbar_arrive_expect_tx(&sh.bar[xb], (uint32_t)(CL * kSmpWarps * 16));
        if (lane < CL)
          st_async4(r_recv + (uint32_t)(((xb * kSmpMaxCL + rank) * kSmpWarps + warp) * 16), d.hi, d.lo, 0.f, 0.f,
                    r_bar + 8u * xb);
        exchange_wait();
        if (*aborted) goto walk_end;
        src_x = xb;
        src_scaled = true;
        R = gather_sum(xb, false);
      }
      const Df T = df_norm(df_mul1(R, p.u_sample[(int64_t)b * n_max + node]));
      // (CTA, warp) level: lane holds the 8 partials of CTA part_r, warps h*8 .. h*8+7
      Df P[kSmpWarps / 2];
      {
        const float f = part_r < CL && !src_scaled ? sh.rk[warp][part_r].x : 1.f;
#pragma unroll
        for (int i = 0; i < kSmpWarps / 2; ++i) {
          P[i] = Df{0.f, 0.f};
          if (part_r < CL) {
            const float4 v = sh.recv[src_x][part_r][(lane & 1) * 8 + i];
            P[i] = src_scaled ? Df{v.x, v.y} : df_mul1({v.x, v.y}, f);
          }
        }
      }
      Df C[kSmpWarps / 2];  // inclusive prefix within the lane
      C[0] = P[0];
#pragma unroll
      for (int i = 1; i < kSmpWarps / 2; ++i) C[i] = dfp_add(C[i - 1], P[i]);
      Df E = C[kSmpWarps / 2 - 1];  // exclusive scan of the lane totals
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const Df y = df_shfl_up(E, o);
        if (lane >= o) E = dfp_add(E, y);
      }
      E = df_shfl_up(E, 1);
      if (lane == 0) E = Df{0.f, 0.f};
      int first = -1, last_nz = -1;
#pragma unroll
      for (int i = 0; i < kSmpWarps / 2; ++i) {
        if (first < 0 && P[i].hi > 0.f && df_gt(df_norm(dfp_add(E, C[i])), T)) first = i;
        if (P[i].hi > 0.f) last_nz = i;
      }
      const unsigned cross = __ballot_sync(0xffffffffu, first >= 0);
      int L, I;
      if (cross) {
        L = __ffs(cross) - 1;
        I = __shfl_sync(0xffffffffu, first, L);
      } else {  // t at or past the total (rounding): the last non-empty warp
        const unsigned nz = __ballot_sync(0xffffffffu, last_nz >= 0);
        L = nz ? 31 - __clz(nz) : 0;
        I = __shfl_sync(0xffffffffu, last_nz < 0 ? 0 : last_nz, L);
      }
      // mass before (CTA, warp) = (L >> 1, (L & 1) * 8 + I), from lane L
      Df pick{0.f, 0.f};
#pragma unroll
      for (int i = 1; i < kSmpWarps / 2; ++i)
        if (i == I) pick = C[i - 1];
      const Df base = df_shfl(df_norm(dfp_add(E, pick)), L);
      if (rank == (L >> 1) && warp == (L & 1) * 8 + I) {
        // thread level inside the chosen warp, in this CTA's unscaled units
        const float ts = pair_sum(nv);
        Df inc = df_mul1({ts, 0.f}, mine.x);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const Df y = df_shfl_up(inc, o);
          if (lane >= o) inc = dfp_add(inc, y);
        }
        Df exc = df_shfl_up(inc, 1);
        if (lane == 0) exc = Df{0.f, 0.f};
        const bool crosses = ts > 0.f && df_gt(df_norm(dfp_add(base, inc)), T);
        const unsigned cr = __ballot_sync(0xffffffffu, crosses);
        const unsigned nzt = __ballot_sync(0xffffffffu, ts > 0.f);
        const int kth = cr ? __ffs(cr) - 1 : (nzt ? 31 - __clz(nzt) : 0);
        if (lane == kth) {
          const Df before = df_norm(dfp_add(base, exc));
          const Df rem = df_gt(T, before) ? df_sub(T, before) : Df{0.f, 0.f};
          const float thr = cr ? (rem.hi + rem.lo) / mine.x : INFINITY;
          float run = 0.f;
          int found = -1, lastv = -1;
#pragma unroll
          for (int e = 0; e < EPT; ++e) {
            run += nv[e];
            if (nv[e] > 0.f) {
              lastv = e;
              if (found < 0 && run > thr) found = e;
            }
          }
          const int e = found >= 0 ? found : lastv;
          bonus = e >= 0 ? t0 + e : -1;
          bonus_writer = 1;
        }
      }
      best = node;
      break;
    }
  walk_end:;
  }

  // ---- outputs, after the previous kernel: the bonus by the thread that drew
  // it, everything else by thread 0 of rank 0.  A request flagged on entry, or
  // with an invalid tree, gets an empty path.  Status bits are OR-ed after every
  // CTA has read the entry value.
  griddep_wait();
  const int st_in = p.status[b];
  int32_t* pn = p.path_nodes + (int64_t)b * n_max;
  int32_t* ot = p.out_tokens + (int64_t)b * (n_max + 1);
  int len_path = 0;
  for (int j = best; j != 0; j = sh.tr.par[j]) ++len_path;
  if (st_in != 0 || bad != 0) {
    if (rank == 0) {
      if (tid == 0) p.accept_len[b] = 0;
      for (int k = tid; k < n_max; k += kSmpThreads) pn[k] = -1;
      for (int k = tid; k <= n_max; k += kSmpThreads) ot[k] = -1;
    }
  } else {
    if (bonus_writer) ot[len_path] = bonus;
    if (rank == 0 && tid == 0) {
      int k = len_path;
      for (int j = best; j != 0; j = sh.tr.par[j]) {
        pn[k] = j;
        ot[k - 1] = sh.tr.tok[j];
        --k;
      }
      pn[0] = 0;
      for (int k2i = len_path + 1; k2i < n_max; ++k2i) pn[k2i] = -1;
      for (int k2i = len_path + 1; k2i <= n_max; ++k2i) ot[k2i] = -1;
      p.accept_len[b] = len_path;
    }
  }
  cluster_arrive();  // no CTA exits while others may still push into it
  cluster_wait();
  if (tid == 0) {
    if (st_in == 0 && bad > 0 && rank == 0) atomicOr(p.status + b, bad);
    if (sh.timed_out) atomicOr(p.status + b, TV_DEV_TIMEOUT);
  }
}

// ---------------------------------------------------------------- host side
template <int EPT, bool kWor>
const void* sample_fn() {
  return (const void*)accept_sample_kernel<EPT, kWor>;
}

constexpr int kEpts[4] = {8, 16, 24, 32};

// clusters of `cl` CTAs of kernel `f` resident at once (cached per context)
int sample_active_clusters(int ei, bool wor, int cl) {
  static int known[2][4][kSmpMaxCL + 1] = {};  // plus 1; 0 = unknown
  static unsigned long long ctx_of = 0;
  unsigned long long ctx = 0;
  if (current_context_id(&ctx) != cudaSuccess) return -1;
  if (ctx == 0 || ctx != ctx_of) {
    for (auto& x : known)
      for (auto& y : x)
        for (int& z : y) z = 0;
    ctx_of = ctx;
  }
  int& slot = known[wor ? 1 : 0][ei][cl];
  if (slot == 0) {
    const void* f = nullptr;
    switch (ei * 2 + (wor ? 1 : 0)) {
      case 0: f = sample_fn<8, false>(); break;
      case 1: f = sample_fn<8, true>(); break;
      case 2: f = sample_fn<16, false>(); break;
      case 3: f = sample_fn<16, true>(); break;
      case 4: f = sample_fn<24, false>(); break;
      case 5: f = sample_fn<24, true>(); break;
      case 6: f = sample_fn<32, false>(); break;
      default: f = sample_fn<32, true>(); break;
    }
    if (cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cl);
    cfg.blockDim = dim3(kSmpThreads);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, f, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    slot = n + 1;
  }
  return slot - 1;
}

template <int EPT, bool kWor>
cudaError_t launch_sample(const SampleParams& p, int B, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B * p.cl);
  cfg.blockDim = dim3(kSmpThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, accept_sample_kernel<EPT, kWor>, p);
}

}  // namespace

// Entries per thread and cluster size: the fewest entries per thread (most
// CTAs per request) whose clusters for the whole batch are resident at once;
// when none is, the most entries per thread (fewest CTAs, fewest waves).
int launch_accept_sample(const float* target, const float* draft, const int32_t* tokens, const int32_t* parents,
                         const int32_t* n_nodes, const float* u_accept, const float* u_sample, int B, int n_max,
                         int V, float temperature, bool without_replacement, int32_t* accept_len,
                         int32_t* path_nodes, int32_t* out_tokens, int32_t* status, cudaStream_t stream) {
  TV_REQUIRE(V <= kSampleMaxV, TV_ERR_UNSUPPORTED,
             "tv_tree_accept: V = %d too large for on-chip sampling (max %d)", V, kSampleMaxV);
  int ei = -1, cl = 0;
  for (int i = 0; i < 4; ++i) {
    const int c = (V + kSmpThreads * kEpts[i] - 1) / (kSmpThreads * kEpts[i]);
    if (c > kSmpMaxCL) continue;
    const int n = sample_active_clusters(i, without_replacement, c);
    TV_REQUIRE(n >= 0, TV_ERR_CUDA, "tv_tree_accept: cluster occupancy query failed");
    if (n >= B) {
      ei = i;
      cl = c;
      break;
    }
  }
  if (ei < 0) {
    ei = 3;
    cl = (V + kSmpThreads * kEpts[3] - 1) / (kSmpThreads * kEpts[3]);
  }
  TV_REQUIRE((int64_t)B * cl < (1ll << 31), TV_ERR_UNSUPPORTED, "tv_tree_accept: B too large");
  SampleParams p;
  p.target = target;
  p.draft = draft;
  p.tokens = tokens;
  p.parents = parents;
  p.n_nodes = n_nodes;
  p.u_accept = u_accept;
  p.u_sample = u_sample;
  p.n_max = n_max;
  p.V = V;
  p.cl = cl;
  p.chunk = kSmpThreads * kEpts[ei];
  p.k2 = (float)(1.4426950408889634 / (double)temperature);
  p.accept_len = accept_len;
  p.path_nodes = path_nodes;
  p.out_tokens = out_tokens;
  p.status = status;
  cudaError_t e;
  switch (ei * 2 + (without_replacement ? 1 : 0)) {
    case 0: e = launch_sample<8, false>(p, B, stream); break;
    case 1: e = launch_sample<8, true>(p, B, stream); break;
    case 2: e = launch_sample<16, false>(p, B, stream); break;
    case 3: e = launch_sample<16, true>(p, B, stream); break;
    case 4: e = launch_sample<24, false>(p, B, stream); break;
    case 5: e = launch_sample<24, true>(p, B, stream); break;
    case 6: e = launch_sample<32, false>(p, B, stream); break;
    default: e = launch_sample<32, true>(p, B, stream); break;
  }
  TV_CUDA_CHECK(e);
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
}

}  // namespace tv
