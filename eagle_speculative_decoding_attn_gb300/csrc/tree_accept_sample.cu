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
  int n_max, V, cl;
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
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// arrival that orders no memory operation (the loads in flight keep going)
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// Commands the controller (warp 0) hands to every warp of its CTA.
enum : int { kCmdPass = 0, kCmdResum = 1, kCmdNode = 2, kCmdBonus = 3, kCmdEnd = 4 };

struct __align__(16) SmpShared {
  float tsum[2][kSmpThreads];            // exchange x: per-thread target (residual) sums, unscaled
  float tsumq[kSmpThreads];              // per-thread draft sums of the exchange being formed
  float4 recv[2][kSmpMaxCL];             // exchange x: every CTA's totals (hi, lo, hi, lo)
  float2 recv_m[2][kSmpMaxCL];           // node visit v: every CTA's maxima (target, draft)
  float2 recv_kid[2][kMaxNodes];         // node visit v: the children's (e_t, e_q), by child position
  float4 rk[kSmpMaxCL];                  // per CTA (alpha, beta, beta / alpha, -) of the node visit
  int2 wmax[2][kSmpWarps];
  uint64_t bar[2];
  AccTree tr;
  // controller -> warps (written before the named barrier that publishes them)
  int cmd;      // kCmd*
  int node;     // kCmdNode: the accepted child
  int xtok;     // kCmdPass: the token this pass rejects (left out of the draft sum)
  int ftok;     // without replacement: token to freeze first, -1 for none
  float c;      // kCmdPass / kCmdResum / kCmdBonus: residual coefficient
  float fc;     // coefficient of the freeze
  int bthr;     // kCmdBonus: the thread of this CTA that draws, -1 for none
  float bthv;   // ... and its threshold (unscaled units; +inf: take its last non-zero entry)
  int timed_out;
};

// Issues the loads of this thread's EPT consecutive entries of a row, from
// token t0.  Entries past V load an in-range entry instead (no select waits on
// the data here); pad_slice turns them into -inf where the values are first used.
template <int EPT>
__device__ __forceinline__ void load_slice(const float* row, int t0, int V, float (&v)[EPT]) {
  if ((V & 3) == 0) {  // rows 16-byte aligned, groups of four never straddle V
#pragma unroll
    for (int i = 0; i < EPT / 4; ++i) {
      const int t = t0 + 4 * i < V ? t0 + 4 * i : 0;
      const float4 x = __ldcs(reinterpret_cast<const float4*>(row + t));
      v[4 * i] = x.x;
      v[4 * i + 1] = x.y;
      v[4 * i + 2] = x.z;
      v[4 * i + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPT; ++i) v[i] = __ldcs(row + (t0 + i < V ? t0 + i : 0));
  }
}
template <int EPT>
__device__ __forceinline__ void pad_slice(int t0, int V, float (&v)[EPT]) {
  if (t0 + EPT > V) {
#pragma unroll
    for (int i = 0; i < EPT; ++i)
      if (t0 + i >= V) v[i] = -INFINITY;
  }
}

// Packed fp32 pairs (two lanes of one 64-bit register, sm_100 family).
__device__ __forceinline__ uint64_t pk(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 upk(uint64_t r) {
  float2 f;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(r));
  return f;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// sum over e of max(0, a[e] - g q[e]): one packed fma per two entries, each
// residual rounded once (the same value as fmaxf(0, fmaf(-g, q, a))), pairs
// summed by packed adds in a fixed tree, then the two halves
template <int EPT>
__device__ __forceinline__ float residual_sum(const float (&a)[EPT], const float (&q)[EPT], float g) {
  static_assert(EPT % 4 == 0, "entries per thread come in fours");
  const uint64_t ng = pk(-g, -g);
  uint64_t s[EPT / 2];
#pragma unroll
  for (int i = 0; i < EPT / 2; ++i) {
    const float2 r = upk(fma2(ng, pk(q[2 * i], q[2 * i + 1]), pk(a[2 * i], a[2 * i + 1])));
    s[i] = pk(fmaxf(0.f, r.x), fmaxf(0.f, r.y));
  }
#pragma unroll
  for (int w = 1; w < EPT / 2; w <<= 1)
#pragma unroll
    for (int i = 0; i + w < EPT / 2; i += 2 * w) s[i] = add2(s[i], s[i + w]);
  const float2 t = upk(s[0]);
  return t.x + t.y;
}

template <int EPT, bool kWor>
__global__ void __launch_bounds__(kSmpThreads, 1) accept_sample_kernel(const SampleParams p) {
  constexpr int kChunk = kSmpThreads * EPT;  // vocabulary entries per CTA
  __shared__ SmpShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int CL = p.cl;
  const int rank = (int)cluster_ctarank();
  const int b = blockIdx.x / CL;
  const int n_max = p.n_max, V = p.V;
  const int t0 = rank * kChunk + tid * EPT;           // this thread's first token
  const int wbase = rank * kChunk + warp * 32 * EPT;  // this warp's first token
  const float k2 = p.k2;

  // Everything up to the outputs reads only inputs (tree, tokens, logits,
  // uniforms) and writes nothing global, so it runs while the previous kernel
  // finishes.  Barrier setup first, published to the cluster by a releasing
  // arrival made before any load is in flight (so it waits for none); then the
  // tree's loads and the root's rows.
  if (tid == 0) {
    mbar_init(&sh.bar[0], 1);
    mbar_init(&sh.bar[1], 1);
    fence_barrier_init();  // for the bytes other CTAs complete on them
    sh.timed_out = 0;
  }
  cluster_arrive_release();
  const AccTreeIn tin = acc_tree_load(p.parents, p.tokens, p.u_accept, p.u_sample, p.n_nodes, b, n_max);
  float a[EPT], q[EPT];
  load_slice<EPT>(p.target + (int64_t)b * n_max * V, t0, V, a);
  load_slice<EPT>(p.draft + (int64_t)b * n_max * V, t0, V, q);
  const int bad = acc_tree_build(sh.tr, tin, n_max, V);
  // remote addresses in CTA `lane` (lanes 0..CL-1 push to the CTA of their index)
  const uint32_t tgt = lane < CL ? (uint32_t)lane : 0u;
  const uint32_t r_recv = mapa_shared(smem_u32(&sh.recv[0][0]), tgt);
  const uint32_t r_recvm = mapa_shared(smem_u32(&sh.recv_m[0][0]), tgt);
  const uint32_t r_kid = mapa_shared(smem_u32(&sh.recv_kid[0][0]), tgt);
  const uint32_t r_bar = mapa_shared(smem_u32(&sh.bar[0]), tgt);
  cluster_wait();

  int node = 0;
  int bonus_writer = 0, bonus = -1;
  int st_pre = -1;  // the status word once read (after the previous kernel)
  if (bad == 0) {  // uniform across the cluster
    int xb = 0, vp = 0;  // exchange buffer, node-visit buffer (same in every warp)
    // ---- controller state (warp 0; identical in every CTA).  Lane j holds
    // child j (and j + 32) of the node: token, u_accept, current (e_t, e_q) in
    // its owner CTA's units; lane r < CL holds CTA r's alpha, beta, beta / alpha.
    uint32_t phase = 0;  // bit x: parity of bar[x]
    float c = 0.f;       // residual coefficient of the current distribution
    float c_try = 0.f;   // ... of the pass in flight
    Df R{0.f, 0.f};      // current residual mass (global scale)
    Df Sq{0.f, 0.f};     // current draft mass (global scale)
    float inv_sq = 0.f;  // 1 / Sq
    float us = 0.f;      // u_sample of the node
    int k = 0, nk = 0;   // child under test, children of the node
    int src_x = 0, src_age = 0;  // exchange holding the current distribution's sums, exchanges since
    bool src_scaled = false;     // its CTA totals are weighted by alpha already (pass totals are)
    int cx[2] = {-1, -1};
    float cu[2] = {0.f, 0.f}, ca[2] = {0.f, 0.f}, cq[2] = {0.f, 0.f};
    float ral = 0.f, rbe = 0.f, rrho = 0.f;

    // controller: this CTA's total of the per-thread values v[0..511], in a
    // fixed order (lane l takes threads l, l + 32, ...)
    auto cta_sum = [&](const float* v) {
      Df s[kSmpWarps];
#pragma unroll
      for (int i = 0; i < kSmpWarps; ++i) s[i] = Df{v[i * 32 + lane], 0.f};
#pragma unroll
      for (int w = 1; w < kSmpWarps; w <<= 1)
#pragma unroll
        for (int i = 0; i + w < kSmpWarps; i += 2 * w) s[i] = dfp_add(s[i], s[i + w]);
      return warp_sum(s[0]);
    };
    // controller: push this CTA's totals (d0, d1) into slot `rank` of every CTA
    auto push_totals = [&](Df d0, Df d1) {
      if (lane < CL)
        st_async4(r_recv + (uint32_t)((xb * kSmpMaxCL + rank) * 16), d0.hi, d0.lo, d1.hi, d1.lo,
                  r_bar + 8u * (uint32_t)xb);
    };
    // controller: wait for exchange xb; false (in every lane) when a wait gave up
    auto ctl_wait = [&]() {
      const bool ok = __all_sync(0xffffffffu, mbar_wait_cluster(&sh.bar[xb], (phase >> xb) & 1u, &sh.timed_out));
      phase ^= 1u << xb;
      if (!ok && lane == 0) sh.timed_out = 1;
      return ok;
    };
    // controller: sum of every CTA's totals of exchange x (first or second
    // double-float), optionally weighted by alpha_r (first) or beta_r (second)
    auto gather_sum = [&](int x, bool second, bool scale) {
      Df s{0.f, 0.f};
      if (lane < CL) {
        const float4 v = sh.recv[x][lane];
        s = second ? Df{v.z, v.w} : Df{v.x, v.y};
        if (scale) s = df_mul1(s, second ? rbe : ral);
      }
#pragma unroll
      for (int o = kSmpMaxCL / 2; o; o >>= 1) s = dfp_add(s, df_shfl_xor(s, o));
      return df_norm(df_shfl(s, 0));
    };
    // child j's slot value from its lane
    auto kid = [&](const float (&v)[2], int j) { return __shfl_sync(0xffffffffu, j >= 32 ? v[1] : v[0], j & 31); };
    auto kidi = [&](const int (&v)[2], int j) { return __shfl_sync(0xffffffffu, j >= 32 ? v[1] : v[0], j & 31); };
    // controller: the bonus draw's position.  Over the CTAs in token order, the
    // first whose running mass exceeds t = u_sample * R; inside that CTA (its
    // controller only) the thread, from the per-thread sums of the source
    // exchange, and that thread's threshold in this CTA's unscaled units
    auto ctl_bonus_scan = [&]() {
      const Df T = df_norm(df_mul1(R, us));
      Df P{0.f, 0.f};
      if (lane < CL) {
        const float4 v = sh.recv[src_x][lane];
        P = src_scaled ? Df{v.x, v.y} : df_mul1({v.x, v.y}, ral);
      }
      Df inc = P;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const Df y = df_shfl_up(inc, o);
        if (lane >= o) inc = dfp_add(inc, y);
      }
      Df exc = df_shfl_up(inc, 1);
      if (lane == 0) exc = Df{0.f, 0.f};
      const unsigned cr = __ballot_sync(0xffffffffu, P.hi > 0.f && df_gt(df_norm(inc), T));
      const unsigned nz = __ballot_sync(0xffffffffu, P.hi > 0.f);
      const int rs = cr ? __ffs(cr) - 1 : (nz ? 31 - __clz(nz) : 0);  // t past the total: last non-empty CTA
      int bthr = -1;
      float bthv = INFINITY;
      if (rs == rank) {
        const Df base_r = df_shfl(df_norm(exc), rs);
        const float al = __shfl_sync(0xffffffffu, ral, rank);
        // lane l: threads 16 l .. 16 l + 15, running sums in unscaled fp32
        float C[16];
        {
          const float4* v4 = reinterpret_cast<const float4*>(&sh.tsum[src_x][16 * lane]);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 w = v4[i];
            C[4 * i] = w.x;
            C[4 * i + 1] = w.y;
            C[4 * i + 2] = w.z;
            C[4 * i + 3] = w.w;
          }
        }
#pragma unroll
        for (int i = 1; i < 16; ++i) C[i] += C[i - 1];  // a thread is non-empty where the running sum grows
        Df E = df_mul1({C[15], 0.f}, al);  // exclusive scan of the lane totals (global scale)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const Df y = df_shfl_up(E, o);
          if (lane >= o) E = dfp_add(E, y);
        }
        E = df_shfl_up(E, 1);
        if (lane == 0) E = Df{0.f, 0.f};
        // this lane's threshold in unscaled units: (t - base_r - E) / alpha
        const Df before = df_norm(dfp_add(base_r, E));
        float thr = 0.f;
        if (df_gt(T, before)) {
          const Df d = df_sub(T, before);
          thr = (d.hi + d.lo) / al;
        }
        int first = -1, last_nz = -1;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const bool grows = C[i] > (i ? C[i - 1] : 0.f);
          if (first < 0 && grows && C[i] > thr) first = i;
          if (grows) last_nz = i;
        }
        const unsigned cl2 = __ballot_sync(0xffffffffu, first >= 0);
        const unsigned nz2 = __ballot_sync(0xffffffffu, last_nz >= 0);
        const bool found = cl2 != 0 && cr != 0;
        const int L = cl2 ? __ffs(cl2) - 1 : (nz2 ? 31 - __clz(nz2) : 0);
        const int I = __shfl_sync(0xffffffffu, cl2 ? first : (last_nz < 0 ? 0 : last_nz), L);
        float prev = 0.f;
#pragma unroll
        for (int i = 1; i < 16; ++i)
          if (i == I) prev = C[i - 1];
        bthr = 16 * L + I;
        bthv = found ? __shfl_sync(0xffffffffu, thr - prev, L) : INFINITY;
      }
      if (lane == 0) {
        sh.bthr = bthr;
        sh.bthv = bthv;
      }
    };
    // controller: test child k; the next command
    auto ctl_next = [&](int ftok, float fc) {
      int cmd = kCmdBonus, nxt = 0, xtok = -1;
      if (k < nk) {
        const int x = kidi(cx, k);
        const float u = kid(cu, k), va = kid(ca, k), vq = kid(cq, k);
        const int o = x / kChunk;
        const float al = __shfl_sync(0xffffffffu, ral, o), be = __shfl_sync(0xffffffffu, rbe, o);
        const float rho = __shfl_sync(0xffffffffu, rrho, o);
        const float pn = al * fmaxf(0.f, fmaf(-(c * rho), vq, va));  // p(x) = pn / R
        const float qn = be * vq;                                     // q(x) = qn / Sq
        // u q(x) < p(x), multiplied through by R Sq > 0 (q = 0 when the draft is empty)
        const bool acc = Sq.hi > 0.f ? (u * qn) * R.hi < pn * Sq.hi : pn > 0.f;
        if (acc) {
          cmd = kCmdNode;
          nxt = sh.tr.kids[sh.tr.kid_off[node] + k];
        } else {  // rejected: the next residual max(0, e_t - c' e_q), c' = c + R / S_q
          cmd = kCmdPass;
          c_try = Sq.hi > 0.f ? fmaf(R.hi, inv_sq, c) : c;
          xtok = x;
        }
      } else if (src_age > 1) {
        // the sums of the current distribution were overwritten (an all-zero
        // residual kept p twice in a row): sum them again first
        cmd = kCmdResum;
        c_try = c;
      } else {
        c_try = c;
        ctl_bonus_scan();
      }
      if (lane == 0) {
        sh.cmd = cmd;
        sh.node = nxt;
        sh.xtok = xtok;
        sh.c = c_try;
        sh.ftok = ftok;
        sh.fc = fc;
      }
    };
    // without replacement: the owner of token x leaves it out of the draft and
    // keeps its residual weight under coefficient cf (same formula as the pass)
    auto freeze = [&](int x, float cf, float rho) {
      if (kWor && x >= 0) {
        const int xe = x - t0;
        if ((unsigned)xe < (unsigned)EPT) {
          const float g = cf * rho;
#pragma unroll
          for (int e = 0; e < EPT; ++e)
            if (e == xe) {
              a[e] = fmaxf(0.f, fmaf(-g, q[e], a[e]));
              q[e] = 0.f;
            }
        }
      }
    };

    for (;;) {
      // ================================ node visit: this CTA's maxima
      pad_slice<EPT>(t0, V, a);
      pad_slice<EPT>(t0, V, q);
      {
        const int it = __reduce_max_sync(0xffffffffu, f2ord(pair_max(a)));
        const int iq = __reduce_max_sync(0xffffffffu, f2ord(pair_max(q)));
        if (lane == 0) sh.wmax[vp][warp] = make_int2(it, iq);
      }
      named_bar_sync(1, kSmpThreads);
      float mt, mq;
      {
        const int2 w = sh.wmax[vp][lane & (kSmpWarps - 1)];
        mt = ord2f(__reduce_max_sync(0xffffffffu, w.x));
        mq = ord2f(__reduce_max_sync(0xffffffffu, w.y));
        if (mt == -INFINITY) mt = 0.f;  // an all-padding slice (weights 0)
        if (mq == -INFINITY) mq = 0.f;
      }
      // exponentiate against the CTA maxima; per-thread sums (the target's in
      // the residual pass's order: it is the residual with coefficient 0)
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        a[e] = exp2f((a[e] - mt) * k2);
        q[e] = exp2f((q[e] - mq) * k2);
      }
      sh.tsum[xb][tid] = residual_sum(a, q, 0.f);
      sh.tsumq[tid] = pair_sum(q);
      const int k_beg = sh.tr.kid_off[node];
      nk = sh.tr.kid_off[node + 1] - k_beg;
      // the children's weights, pushed by their owner warps
      for (int j0 = 0; j0 < nk; j0 += 32) {
        const int j = j0 + lane;
        const int x = j < nk ? sh.tr.tok[sh.tr.kids[k_beg + j]] : -1;
        const unsigned own = __ballot_sync(0xffffffffu, j < nk && (unsigned)(x - wbase) < (unsigned)(32 * EPT));
        for (unsigned m = own; m; m &= m - 1) {
          const int src = __ffs(m) - 1;
          const int xx = __shfl_sync(0xffffffffu, x, src);
          const int ol = (xx - wbase) / EPT, e = (xx - wbase) - ol * EPT;
          const float ax = __shfl_sync(0xffffffffu, reg_at(a, e), ol);
          const float qx = __shfl_sync(0xffffffffu, reg_at(q, e), ol);
          if (lane < CL)
            st_async2(r_kid + (uint32_t)((vp * kMaxNodes + j0 + src) * 8), ax, qx, r_bar + 8u * (uint32_t)xb);
        }
      }
      named_bar_sync(1, kSmpThreads);
      if (warp == 0) {
        // publish this CTA's totals and maxima (every CTA expects CL of each and
        // one 8-byte push per child)
        const Df st = cta_sum(sh.tsum[xb]);
        const Df sq = cta_sum(sh.tsumq);
        if (lane == 0) mbar_arrive_expect_tx(&sh.bar[xb], (uint32_t)(CL * (16 + 8) + nk * 8));
        push_totals(st, sq);
        if (lane < CL)
          st_async2(r_recvm + (uint32_t)((vp * kSmpMaxCL + rank) * 8), mt, mq, r_bar + 8u * (uint32_t)xb);
        // the children's tokens and uniforms, and u_sample, do not wait for the exchange
        us = sh.tr.us[node];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = lane + 32 * h;
          const int ch = j < nk ? sh.tr.kids[k_beg + j] : 0;
          cx[h] = j < nk ? sh.tr.tok[ch] : -1;
          cu[h] = sh.tr.ua[ch];
        }
        if (!ctl_wait()) {
          if (lane == 0) sh.cmd = kCmdEnd;
        } else {
          // per-CTA weights alpha_r, beta_r against the global maxima
          const float2 m = lane < CL ? sh.recv_m[vp][lane] : make_float2(-INFINITY, -INFINITY);
          const float Mt = ord2f(__reduce_max_sync(0xffffffffu, f2ord(m.x)));
          const float Mq = ord2f(__reduce_max_sync(0xffffffffu, f2ord(m.y)));
          ral = lane < CL ? exp2f((m.x - Mt) * k2) : 0.f;
          rbe = lane < CL ? exp2f((m.y - Mq) * k2) : 0.f;
          rrho = ral > 0.f ? rbe * __frcp_rn(ral) : 0.f;
          if (lane < CL) sh.rk[lane] = make_float4(ral, rbe, rrho, 0.f);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int j = lane + 32 * h;
            const float2 kv = j < nk ? sh.recv_kid[vp][j] : make_float2(0.f, 0.f);
            ca[h] = kv.x;
            cq[h] = kv.y;
          }
          R = gather_sum(xb, false, true);
          Sq = gather_sum(xb, true, true);
          inv_sq = Sq.hi > 0.f ? __frcp_rn(Sq.hi) : 0.f;
          c = 0.f;
          k = 0;
          src_x = xb;
          src_scaled = false;
          src_age = 0;
          ctl_next(-1, 0.f);
        }
      }
      xb ^= 1;
      vp ^= 1;
      named_bar_sync(1, kSmpThreads);
      int cmd = sh.cmd;

      // ================================ residual passes
      while (cmd == kCmdPass || cmd == kCmdResum) {
        const float4 mine = sh.rk[rank];  // this CTA's (alpha, beta, beta / alpha)
        freeze(sh.ftok, sh.fc, mine.z);
        const float g = sh.c * mine.z;
        sh.tsum[xb][tid] = residual_sum(a, q, g);
        if (kWor) {
          const int xe = cmd == kCmdPass ? sh.xtok - t0 : -1;  // the rejected token's register, if here
          float zq[EPT];
#pragma unroll
          for (int e = 0; e < EPT; ++e) zq[e] = e == xe ? 0.f : q[e];
          sh.tsumq[tid] = pair_sum(zq);
        }
        named_bar_sync(1, kSmpThreads);
        if (warp == 0) {
          const Df dz = df_mul1(cta_sum(sh.tsum[xb]), mine.x);
          Df dq{0.f, 0.f};
          if (kWor) dq = df_mul1(cta_sum(sh.tsumq), mine.y);
          if (lane == 0) mbar_arrive_expect_tx(&sh.bar[xb], (uint32_t)(CL * 16));
          push_totals(dz, dq);
          if (!ctl_wait()) {
            if (lane == 0) sh.cmd = kCmdEnd;
          } else if (cmd == kCmdResum) {
            R = gather_sum(xb, false, false);
            src_x = xb;
            src_scaled = true;
            src_age = 0;
            ctl_next(-1, 0.f);
          } else {
            const Df Z = gather_sum(xb, false, false);
            const bool kept = !(Z.hi > 0.f);  // an all-zero residual keeps p
            ++src_age;
            if (!kept) {
              src_x = xb;
              src_scaled = true;
              src_age = 0;
            }
            const float c_eff = kept ? c : c_try;
            int x = -1;
            if (kWor) {
              // x leaves the draft; every child with token x keeps x's weight of the
              // distribution now current
              x = kidi(cx, k);
              const float va = kid(ca, k), vq = kid(cq, k);
              const float rho = __shfl_sync(0xffffffffu, rrho, x / kChunk);
              const float fz = fmaxf(0.f, fmaf(-(c_eff * rho), vq, va));
#pragma unroll
              for (int h = 0; h < 2; ++h)
                if (cx[h] == x) {
                  ca[h] = fz;
                  cq[h] = 0.f;
                }
              Sq = gather_sum(xb, true, false);
              inv_sq = Sq.hi > 0.f ? __frcp_rn(Sq.hi) : 0.f;
            }
            if (!kept) {
              c = c_try;
              R = Z;
            }
            ++k;
            ctl_next(x, c_eff);
          }
        }
        xb ^= 1;
        named_bar_sync(1, kSmpThreads);
        cmd = sh.cmd;
      }
      if (cmd == kCmdNode) {
        node = sh.node;
        load_slice<EPT>(p.target + ((int64_t)b * n_max + node) * V, t0, V, a);
        load_slice<EPT>(p.draft + ((int64_t)b * n_max + node) * V, t0, V, q);
        continue;
      }
      // the previous kernel has long finished: fetch the status word now, so its
      // load overlaps the bonus draw
      griddep_wait();
      st_pre = p.status[b];
      if (cmd == kCmdBonus && tid == sh.bthr) {
        // ---- bonus token: the first entry of this thread whose running residual
        // weight (unscaled) exceeds the threshold; the last non-zero one when the
        // rounding left none
        const float4 mine = sh.rk[rank];
        freeze(sh.ftok, sh.fc, mine.z);
        const float g = sh.c * mine.z;
        const float thr = sh.bthv;
        float run = 0.f;
        int found = -1, lastv = -1;
#pragma unroll
        for (int e = 0; e < EPT; ++e) {
          const float nv = fmaxf(0.f, fmaf(-g, q[e], a[e]));
          run += nv;
          if (nv > 0.f) {
            lastv = e;
            if (found < 0 && run > thr) found = e;
          }
        }
        const int e = found >= 0 ? found : lastv;
        bonus = e >= 0 ? t0 + e : -1;
        bonus_writer = 1;
      }
      break;
    }
  }

  // ---- outputs, after the previous kernel: the bonus by the thread that drew
  // it, the rest by rank 0.  A request flagged on entry, or with an invalid
  // tree, gets an empty path.  Status bits are OR-ed after every CTA has read
  // the entry value (the cluster barrier), and no CTA exits while another may
  // still push into it.
  if (st_pre < 0) {
    griddep_wait();
    st_pre = p.status[b];
  }
  const int st_in = st_pre;  // consumed below, before this thread's arrival completes its part
  cluster_arrive_relaxed();
  int32_t* pn = p.path_nodes + (int64_t)b * n_max;
  int32_t* ot = p.out_tokens + (int64_t)b * (n_max + 1);
  if (st_in != 0 || bad != 0) {
    if (rank == 0) {
      if (tid == 0) p.accept_len[b] = 0;
      for (int i = tid; i < n_max; i += kSmpThreads) pn[i] = -1;
      for (int i = tid; i <= n_max; i += kSmpThreads) ot[i] = -1;
    }
  } else {
    int len_path = 0;
    for (int j = node; j != 0; j = sh.tr.par[j]) ++len_path;
    if (bonus_writer) ot[len_path] = bonus;
    if (rank == 0) {
      // thread i < len_path writes path entry i + 1; the rest fill -1
      if (tid < len_path) {
        int j = node;
        for (int s = len_path - 1; s > tid; --s) j = sh.tr.par[j];
        pn[tid + 1] = j;
        ot[tid] = sh.tr.tok[j];
      }
      if (tid == 0) {
        pn[0] = 0;
        p.accept_len[b] = len_path;
        if (sh.timed_out) ot[len_path] = -1;
      }
      for (int i = len_path + 1 + tid; i < n_max; i += kSmpThreads) pn[i] = -1;
      for (int i = len_path + 1 + tid; i <= n_max; i += kSmpThreads) ot[i] = -1;
    }
  }
  cluster_wait();
  if (tid == 0) {
    if (st_in == 0 && bad > 0 && rank == 0) atomicOr(p.status + b, bad);
    if (sh.timed_out) atomicOr(p.status + b, TV_DEV_TIMEOUT);
  }
}

// ---------------------------------------------------------------- host side
constexpr int kNumEpt = 5;
constexpr int kEpts[kNumEpt] = {8, 16, 20, 24, 32};
using SampleKernel = void (*)(SampleParams);
// [entries-per-thread index][without replacement]
const SampleKernel kSampleKernels[kNumEpt][2] = {
    {accept_sample_kernel<8, false>, accept_sample_kernel<8, true>},
    {accept_sample_kernel<16, false>, accept_sample_kernel<16, true>},
    {accept_sample_kernel<20, false>, accept_sample_kernel<20, true>},
    {accept_sample_kernel<24, false>, accept_sample_kernel<24, true>},
    {accept_sample_kernel<32, false>, accept_sample_kernel<32, true>},
};

// clusters of `cl` CTAs of the kernel resident at once (cached per context);
// -1 when a CUDA call fails
int sample_active_clusters(int ei, bool wor, int cl) {
  static int known[kNumEpt][2][kSmpMaxCL + 1] = {};  // plus 1; 0 = unknown
  static unsigned long long ctx_of = 0;
  unsigned long long ctx = 0;
  if (current_context_id(&ctx) != cudaSuccess) return -1;
  if (ctx == 0 || ctx != ctx_of) {
    for (auto& x : known)
      for (auto& y : x)
        for (int& z : y) z = 0;
    ctx_of = ctx;
  }
  int& slot = known[ei][wor ? 1 : 0][cl];
  if (slot == 0) {
    const SampleKernel f = kSampleKernels[ei][wor ? 1 : 0];
    if (cudaFuncSetAttribute((const void*)f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return -1;
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
  auto ctas = [&](int ei) { return (V + kSmpThreads * kEpts[ei] - 1) / (kSmpThreads * kEpts[ei]); };
  int ei = -1;
  for (int i = 0; i < kNumEpt; ++i) {
    if (ctas(i) > kSmpMaxCL) continue;
    const int n = sample_active_clusters(i, without_replacement, ctas(i));
    TV_REQUIRE(n >= 0, TV_ERR_CUDA, "tv_tree_accept: cluster occupancy query failed");
    if (n >= B) {
      ei = i;
      break;
    }
  }
  if (ei < 0) ei = kNumEpt - 1;
  const int cl = ctas(ei);
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
  p.k2 = (float)(1.4426950408889634 / (double)temperature);
  p.accept_len = accept_len;
  p.path_nodes = path_nodes;
  p.out_tokens = out_tokens;
  p.status = status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B * cl);
  cfg.blockDim = dim3(kSmpThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  TV_CUDA_CHECK(cudaLaunchKernelEx(&cfg, kSampleKernels[ei][without_replacement ? 1 : 0], p));
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
}

}  // namespace tv
