// tv_tree_expand: one level of dynamic draft-tree construction.
//
// "SGLang EAGLE-2 Speculative Decoding" (Tech Radar), section 2: per expansion
// depth the drafter's distribution is scored by its entropy
// H = -sum_i P(x_i) log P(x_i) (section "Dynamic Tree-Attention Masking"):
// a low-entropy node extends a single branch, a high-entropy node widens the
// tree up to 8 children; beam search then prunes the low branches (sequence
// diagram) and the tree stays within 64 nodes.
//
// Per frontier node f: P = softmax(draft row f), w_f = round(e^H) clamped to
// [1, top_k] (e^H, the perplexity, is the number of equally likely tokens with
// the same entropy), candidates = the w_f most probable tokens with cumulative
// score score_f + log P(token).  The best min(max_new, budget - n_nodes)
// candidates by score (equal scores: lower f, then lower rank) are appended in
// (f, rank) order, so parents precede children and siblings are contiguous.
//
// One launch per level.  A work item is one 8192-logit slice of one frontier
// row; it is reduced to (max, sum e^(x-max), sum e^(x-max)(x-max)) and its 8
// largest logits.  The last item of a request to finish (arrival counter)
// merges the slices of every frontier row, takes the widths and the beam
// selection in shared memory and appends the nodes.  The logits are read once:
// the kernel is bound by HBM.
//
// One CTA per potential item (slice, frontier row, request) loads its slice
// straight into registers (16-byte loads when V is a multiple of 4); four CTAs
// share an SM so that the loads of some overlap the reductions of others.
// (A persistent form that staged slices through a shared-memory ring with the
// bulk-copy engine measured slower: its per-slice reduction, barriers and
// arrival are a serial latency chain that two resident CTAs did not hide.)
#include <cfloat>
#include <climits>
#include <cmath>

#include "tv_common.cuh"

namespace tv {

constexpr int kExpThreads = 256;
constexpr int kExpPerThread = 32;                        // logits per thread and slice
constexpr int kExpSlice = kExpThreads * kExpPerThread;   // 8192
constexpr int kExpTop = 8;                               // widest branching (width <= 8)
constexpr int kSliceCand = 256;                          // threshold candidates of a slice
constexpr int kExpWarps = kExpThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;

struct __align__(16) ExpPart {  // one slice of one draft row
  float m, s, t, pad;           // max, sum e^(x-m), sum e^(x-m)(x-m)
  float v[kExpTop];             // largest logits, descending
  int i[kExpTop];               // their token ids (ascending on equal logits)
};

struct ExpandParams {
  const float* logits;
  int32_t* parents;
  int32_t* tokens;
  float* scores;
  int32_t* n_nodes;
  int32_t* level_start;
  float* entropy;
  int32_t* width;
  int n_max, V, top_k, max_new, budget, max_frontier, n_slices;
  float width_ln[kExpTop];  // width_ln[j] = ln(j + 1/2), rounded once from double: H at or above it gives > j children
  ExpPart* part;      // [B][max_frontier][n_slices]
  int32_t* tickets;   // [B] arrivals of this call (zero between calls)
  int32_t* status;
};

struct ExpShared {
  int wmax_k[kExpWarps];  // order keys of the warps' largest logits
  int wcnt[kExpWarps];    // candidates of each warp
  float red_s[kExpWarps], red_t[kExpWarps];
  float wtop_v[kExpWarps][kExpTop];
  int wtop_i[kExpWarps][kExpTop];
  float top_v[kExpTop];
  int top_i[kExpTop];
  float cand_v[kSliceCand];
  int cand_i[kSliceCand];
  int last;
  // merge of a request
  float row_c[kMaxNodes][kExpTop];
  int row_tok[kMaxNodes][kExpTop];
  int row_w[kMaxNodes];
  int row_off[kMaxNodes + 1];
  float mc[kMaxNodes * kExpTop];
  int mkey[kMaxNodes * kExpTop];
  int sel_cnt[2][kExpWarps];
};

// (v1, i1) ranks before (v2, i2): larger logit, then lower token id.
__device__ __forceinline__ bool top_before(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

__device__ __forceinline__ void top_clear(float (&v)[kExpTop], int (&ix)[kExpTop]) {
#pragma unroll
  for (int k = 0; k < kExpTop; ++k) {
    v[k] = -INFINITY;
    ix[k] = INT_MAX;
  }
}

// Insert (x, j) into a sorted list of the 8 best; returns false when it does
// not enter the list.
__device__ __forceinline__ bool top_insert(float (&v)[kExpTop], int (&ix)[kExpTop], float x, int j) {
  if (!top_before(x, j, v[kExpTop - 1], ix[kExpTop - 1])) return false;
  v[kExpTop - 1] = x;
  ix[kExpTop - 1] = j;
#pragma unroll
  for (int k = kExpTop - 1; k > 0; --k) {
    if (top_before(v[k], ix[k], v[k - 1], ix[k - 1])) {
      const float tv = v[k];
      v[k] = v[k - 1];
      v[k - 1] = tv;
      const int ti = ix[k];
      ix[k] = ix[k - 1];
      ix[k - 1] = ti;
    }
  }
  return true;
}

// The warp's 8 best of the lanes' sorted lists, in every lane (ov, oi).  Each
// round takes the best list head across the warp and pops it from its lane.
__device__ __forceinline__ void warp_top8(float (&v)[kExpTop], int (&ix)[kExpTop], float (&ov)[kExpTop],
                                          int (&oi)[kExpTop]) {
#pragma unroll
  for (int r = 0; r < kExpTop; ++r) {
    float bv = v[0];
    int bi = ix[0];
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      if (top_before(v2, i2, bv, bi)) {
        bv = v2;
        bi = i2;
      }
    }
    ov[r] = bv;
    oi[r] = bi;
    if (v[0] == bv && ix[0] == bi) {  // token ids are unique, sentinels harmless
#pragma unroll
      for (int k = 0; k < kExpTop - 1; ++k) {
        v[k] = v[k + 1];
        ix[k] = ix[k + 1];
      }
      v[kExpTop - 1] = -INFINITY;
      ix[kExpTop - 1] = INT_MAX;
    }
  }
}

// Merge (m2, s2, t2) into (m, s, t); s = 0 marks an empty part.
__device__ __forceinline__ void mst_merge(float& m, float& s, float& t, float m2, float s2, float t2) {
  if (s2 == 0.f) return;
  if (s == 0.f) {
    m = m2;
    s = s2;
    t = t2;
    return;
  }
  const float mn = fmaxf(m, m2);
  const float d1 = m - mn, d2 = m2 - mn;
  const float a1 = ex2_approx(d1 * kLog2e), a2 = ex2_approx(d2 * kLog2e);
  t = a1 * fmaf(d1, s, t) + a2 * fmaf(d2, s2, t2);
  s = a1 * s + a2 * s2;
  m = mn;
}

__device__ __forceinline__ void warp_mst(float& m, float& s, float& t) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float t2 = __shfl_xor_sync(0xffffffffu, t, o);
    mst_merge(m, s, t, m2, s2, t2);
  }
}

// Thread's 32 logits of a slice: element (u, c) is logit lo + 4 * (u * 256 +
// tid) + c, so token ids rise along u and c and equal logits keep the lower id
// first; entries past hi are -inf.
__device__ __forceinline__ int slice_j(int lo, int u, int c) { return lo + 4 * (u * kExpThreads + threadIdx.x) + c; }

// Order key of a float: larger floats have larger (signed) keys.
__device__ __forceinline__ int f2key(float f) {
  const int i = __float_as_int(f);
  return i ^ ((i >> 31) & 0x7fffffff);
}
__device__ __forceinline__ float key2f(int k) { return __int_as_float(k ^ ((k >> 31) & 0x7fffffff)); }

// Sum over the warp, in every lane.
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Reduce one slice (x in registers: the row's logits lo .. hi - 1, at least
// one) to its part: M = the slice's max, sum e^(x-M), sum e^(x-M)(x-M) and its
// 8 largest logits with their token ids; thread 0 stores it at dst (and
// publishes it with a fence before arriving).
//
// Each warp's largest logit is a distinct logit, so with 8 warps the slice's 8
// best are all >= T, the smallest warp maximum: only logits >= T are
// candidates.  Every thread reads M and T from the warps' maxima; the
// candidates are placed by a scan of their counts (no atomics) and ranked
// against each other (larger logit, then lower token id first).
__device__ __forceinline__ void slice_reduce(ExpShared& sh, const float (&x)[kExpPerThread], const float* row,
                                             int lo, int hi, ExpPart* dst) {
  static_assert(kExpWarps == kExpTop, "the threshold is the smallest of 8 warp maxima");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float m4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
  for (int k = 4; k < kExpPerThread; ++k) m4[k & 3] = fmaxf(m4[k & 3], x[k]);
  const int wk = __reduce_max_sync(0xffffffffu, f2key(fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]))));
  if (lane == 0) sh.wmax_k[warp] = wk;
  __syncthreads();
  if (tid == 0) {  // after the barrier: the previous slice's readers of the list are done
#pragma unroll
    for (int k = 0; k < kExpTop; ++k) {
      sh.top_v[k] = -INFINITY;
      sh.top_i[k] = INT_MAX;
    }
  }
  int kmax = INT_MIN, kmin = INT_MAX;
#pragma unroll
  for (int w = 0; w < kExpWarps; ++w) {
    const int k = sh.wmax_k[w];
    kmax = max(kmax, k);
    kmin = min(kmin, k);
  }
  const float M = key2f(kmax), T = key2f(kmin);
  // sums against M in base 2 (d >= -288 keeps e * d finite: e is then 0), and
  // the thread's candidates
  const float ml2 = M * kLog2e;
  float s4[4] = {0.f, 0.f, 0.f, 0.f}, t4[4] = {0.f, 0.f, 0.f, 0.f};
  int cnt = 0;
#pragma unroll
  for (int k = 0; k < kExpPerThread; ++k) {
    const float d = fmaxf(fmaf(x[k], kLog2e, -ml2), -288.f);
    const float e = ex2_approx(d);
    s4[k & 3] += e;
    t4[k & 3] = fmaf(e, d, t4[k & 3]);
    cnt += x[k] >= T && slice_j(lo, k >> 2, k & 3) < hi;
  }
  const float s_w = warp_sum((s4[0] + s4[1]) + (s4[2] + s4[3]));
  const float t_w = warp_sum((t4[0] + t4[1]) + (t4[2] + t4[3]));
  int incl = cnt;  // inclusive scan of the counts over the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) {
    sh.red_s[warp] = s_w;
    sh.red_t[warp] = t_w;
    sh.wcnt[warp] = incl;
  }
  __syncthreads();
  int pos = incl - cnt, nc = 0;
#pragma unroll
  for (int w = 0; w < kExpWarps; ++w) {
    const int c = sh.wcnt[w];
    pos += w < warp ? c : 0;
    nc += c;
  }
  if (nc <= kSliceCand) {
    if (cnt > 0) {
#pragma unroll
      for (int k = 0; k < kExpPerThread; ++k) {
        const int j = slice_j(lo, k >> 2, k & 3);
        if (x[k] >= T && j < hi) {
          sh.cand_v[pos] = x[k];
          sh.cand_i[pos] = j;
          ++pos;
        }
      }
    }
    __syncthreads();
    // a candidate's rank among the candidates; ranks 0..7 are the slice's 8 best
    if (tid < nc) {
      const float v = sh.cand_v[tid];
      const int i = sh.cand_i[tid];
      int rank = 0;
#pragma unroll 4
      for (int c = 0; c < nc; ++c) rank += top_before(sh.cand_v[c], sh.cand_i[c], v, i);
      if (rank < kExpTop) {
        sh.top_v[rank] = v;
        sh.top_i[rank] = i;
      }
    }
  } else {
    // many logits equal to T: exact per-thread lists instead, over the slice
    // read again (rare; the registers of x are free by now)
    float tv_[kExpTop], ov[kExpTop];
    int ti_[kExpTop], oi[kExpTop];
    top_clear(tv_, ti_);
#pragma unroll 1
    for (int u = 0; u < kExpPerThread / 4; ++u)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = slice_j(lo, u, c);
        if (j < hi) top_insert(tv_, ti_, __ldcg(row + j), j);
      }
    warp_top8(tv_, ti_, ov, oi);
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < kExpTop; ++k) {
        sh.wtop_v[warp][k] = ov[k];
        sh.wtop_i[warp][k] = oi[k];
      }
    }
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int k = 0; k < kExpTop; ++k) {
        tv_[k] = lane < kExpWarps ? sh.wtop_v[lane][k] : -INFINITY;
        ti_[k] = lane < kExpWarps ? sh.wtop_i[lane][k] : INT_MAX;
      }
      warp_top8(tv_, ti_, ov, oi);
      if (lane == 0) {
#pragma unroll
        for (int k = 0; k < kExpTop; ++k) {
          sh.top_v[k] = ov[k];
          sh.top_i[k] = oi[k];
        }
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    const float s = warp_sum(lane < kExpWarps ? sh.red_s[lane] : 0.f);
    const float t = warp_sum(lane < kExpWarps ? sh.red_t[lane] : 0.f) * 0.69314718055994531f;  // base 2 -> e
    if (lane == 0) {
      ExpPart r;
      r.m = M;
      r.s = s;
      r.t = t;
      r.pad = 0.f;
#pragma unroll
      for (int k = 0; k < kExpTop; ++k) {
        r.v[k] = sh.top_v[k];
        r.i[k] = sh.top_i[k];
      }
      *dst = r;
    }
  }
}

// Thread 0 (the writer of this CTA's parts) publishes them and arrives `cnt`
// times on request b's counter; returns (block-uniform) whether the request's
// parts are now complete.
__device__ __forceinline__ bool arrive(ExpShared& sh, int32_t* ticket, int cnt, int expected) {
  if (threadIdx.x == 0) {
    __threadfence();
    sh.last = atomicAdd(ticket, cnt) + cnt == expected;
  }
  __syncthreads();
  const bool last = sh.last;
  if (last) __threadfence();
  return last;
}

// The last arrival of request b: merge the parts of its F frontier rows
// (state n, ls), take the widths and the beam cut, append the kept nodes at
// n, n + 1, ...  Returns how many were appended.
__device__ int request_merge(ExpShared& sh, const ExpandParams& p, int b, int n, int ls, int F) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_max = p.n_max;
  float tv_[kExpTop], ov[kExpTop];
  int ti_[kExpTop], oi[kExpTop];
  // warp w takes rows w, w + 8, ...: lanes take the row's slices
  const bool lane_lists = p.n_slices * kExpTop <= 32;
  for (int r = warp; r < F; r += kExpWarps) {
    const ExpPart* src = p.part + ((int64_t)b * p.max_frontier + r) * p.n_slices;
    // every load of the row first (one round trip): the sums of the lane's
    // first slice, its list entry (one per lane when the lists fit the warp)
    // and the node's score
    const int ne = p.n_slices * kExpTop;
    const bool has = lane_lists && lane < ne;
    const ExpPart* pq = src + lane / kExpTop;
    const float v = has ? __ldcg(pq->v + lane % kExpTop) : -INFINITY;
    const int i = has ? __ldcg(pq->i + lane % kExpTop) : INT_MAX;
    const float4 w0 = lane < p.n_slices ? __ldcg(reinterpret_cast<const float4*>(src + lane))
                                        : make_float4(-INFINITY, 0.f, 0.f, 0.f);
    const float sf = p.scores[(int64_t)b * n_max + ls + r];
    float m = w0.x, s = w0.y, t = w0.z;
    for (int q = lane + 32; q < p.n_slices; q += 32) {
      const float4 wq = __ldcg(reinterpret_cast<const float4*>(src + q));
      mst_merge(m, s, t, wq.x, wq.y, wq.z);
    }
    warp_mst(m, s, t);
    const float lz = logf(s);  // log of the normaliser, relative to m
    const float H = lz - t / s;
    int real;
    if (lane_lists) {
      // one list entry per lane, ranked against the others (entries equal in
      // full, the padding of short lists, by lane)
      int rank = 0;
      for (int o = 0; o < ne; ++o) {
        const float vo = __shfl_sync(0xffffffffu, v, o);
        const int io = __shfl_sync(0xffffffffu, i, o);
        rank += top_before(vo, io, v, i) || (vo == v && io == i && o < lane);
      }
      const bool top = has && rank < kExpTop;
      real = __popc(__ballot_sync(0xffffffffu, top && i != INT_MAX));
      if (top) {
        sh.row_c[r][rank] = sf + ((v - m) - lz);
        sh.row_tok[r][rank] = i;
      }
    } else {
      top_clear(tv_, ti_);
      for (int q = lane; q < p.n_slices; q += 32) {
        const float4* w4 = reinterpret_cast<const float4*>(src + q);
        float4 w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) w[k] = __ldcg(w4 + 1 + k);
        const float pv[kExpTop] = {w[0].x, w[0].y, w[0].z, w[0].w, w[1].x, w[1].y, w[1].z, w[1].w};
        const int pi[kExpTop] = {__float_as_int(w[2].x), __float_as_int(w[2].y), __float_as_int(w[2].z),
                                 __float_as_int(w[2].w), __float_as_int(w[3].x), __float_as_int(w[3].y),
                                 __float_as_int(w[3].z), __float_as_int(w[3].w)};
#pragma unroll
        for (int k = 0; k < kExpTop; ++k)
          if (!top_insert(tv_, ti_, pv[k], pi[k])) break;  // the part's list is sorted
      }
      warp_top8(tv_, ti_, ov, oi);
      real = 0;
#pragma unroll
      for (int k = 0; k < kExpTop; ++k) real += oi[k] != INT_MAX;
      if (lane < kExpTop) {
        float vk = ov[0];
        int ik = oi[0];
#pragma unroll
        for (int k = 1; k < kExpTop; ++k)
          if (lane == k) {
            vk = ov[k];
            ik = oi[k];
          }
        sh.row_c[r][lane] = sf + ((vk - m) - lz);
        sh.row_tok[r][lane] = ik;
      }
    }
    if (lane == 0) {
      int w = 1;
      for (int j = 1; j < p.top_k; ++j) w += H >= p.width_ln[j];
      w = min(w, real);
      const int f = ls + r;
      if (p.entropy) p.entropy[(int64_t)b * n_max + f] = H;
      if (p.width) p.width[(int64_t)b * n_max + f] = w;
      sh.row_w[r] = w;
    }
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the widths over the (at most 64) frontier rows
    const int w0 = lane < F ? sh.row_w[lane] : 0;
    const int w1 = lane + 32 < F ? sh.row_w[lane + 32] : 0;
    int i0 = w0, i1 = w1;
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
    const int tot1 = __shfl_sync(0xffffffffu, i1, 31);
    if (lane < F) sh.row_off[lane] = i0 - w0;
    if (lane + 32 < F) sh.row_off[lane + 32] = tot0 + i1 - w1;
    if (lane == 0) sh.row_off[F] = tot0 + tot1;
  }
  __syncthreads();
  const int C = sh.row_off[F];
  for (int a = tid; a < F * kExpTop; a += kExpThreads) {
    const int r = a / kExpTop, k = a % kExpTop;
    if (k < sh.row_w[r]) {
      sh.mc[sh.row_off[r] + k] = sh.row_c[r][k];
      sh.mkey[sh.row_off[r] + k] = a;  // dense order = (row, rank) order
    }
  }
  __syncthreads();
  const int keep = min(min(p.max_new, p.budget - n), C);
  // rank of each candidate by score (equal scores: earlier in (row, rank)
  // order first); the best `keep` are appended in (row, rank) order
  for (int h = 0; h * kExpThreads < C; ++h) {  // C is the same in every thread
    const int d = h * kExpThreads + tid;
    bool sel = false;
    if (d < C) {
      const float c = sh.mc[d];
      int rank = 0;
#pragma unroll 8
      for (int e = 0; e < C; ++e) {
        const float ce = sh.mc[e];
        rank += (ce > c) || (ce == c && e < d);
      }
      sel = rank < keep;
    }
    const unsigned bal = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) sh.sel_cnt[h][warp] = __popc(bal);
    __syncthreads();
    if (sel) {
      int pos = __popc(bal & ((1u << lane) - 1u));
      for (int hh = 0; hh < h; ++hh)
        for (int w = 0; w < kExpWarps; ++w) pos += sh.sel_cnt[hh][w];
      for (int w = 0; w < warp; ++w) pos += sh.sel_cnt[h][w];
      const int key = sh.mkey[d];
      const int r = key / kExpTop, k = key % kExpTop;
      const int64_t o = (int64_t)b * n_max + n + pos;
      p.parents[o] = ls + r;
      p.tokens[o] = sh.row_tok[r][k];
      p.scores[o] = sh.row_c[r][k];
    }
  }
  __syncthreads();  // the merge arrays may be reused by the next request
  return keep;
}

// CTA (slice, frontier row, request).  Every CTA of a request arrives, live or
// not, so the last one runs after every read of that request's state.
__global__ void __launch_bounds__(kExpThreads, 4) tree_expand_kernel(const ExpandParams p) {
  __shared__ ExpShared sh;
  const int sl = blockIdx.x, y = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int n_max = p.n_max, V = p.V;
  griddep_wait();  // no early trigger: the acceptance reads what this kernel writes before its own wait
  const int st = p.status[b];
  const int n = p.n_nodes[b], ls = p.level_start[b];
  const bool ok = st == 0 && n >= 1 && n <= n_max && ls >= 0 && ls <= n;
  const int F = ok ? n - ls : 0;
  const bool work = ok && y < F && F <= p.max_frontier && n < p.budget;

  if (work) {
    // CTAs past the frontier only arrive: their parts are never read
    float x[kExpPerThread];
    const float* row = p.logits + ((int64_t)b * n_max + ls + y) * V;
    const int lo = sl * kExpSlice;
    const int hi = min(V, lo + kExpSlice);
    if ((V & 3) == 0) {
      const float4* r4 = reinterpret_cast<const float4*>(row + lo);
#pragma unroll
      for (int u = 0; u < kExpPerThread / 4; ++u) {
        const int e = 4 * (u * kExpThreads + tid);
        const float4 q = lo + e < hi ? __ldcs(r4 + u * kExpThreads + tid)
                                     : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        x[4 * u] = q.x;
        x[4 * u + 1] = q.y;
        x[4 * u + 2] = q.z;
        x[4 * u + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int u = 0; u < kExpPerThread / 4; ++u)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int j = slice_j(lo, u, c);
          x[4 * u + c] = j < hi ? __ldcs(row + j) : -INFINITY;
        }
    }
    slice_reduce(sh, x, row, lo, hi, p.part + ((int64_t)b * p.max_frontier + y) * p.n_slices + sl);
  }
  if (!arrive(sh, p.tickets + b, 1, p.max_frontier * p.n_slices)) return;

  // ---- the last CTA of request b
  if (!ok || F > p.max_frontier) {
    if (tid == 0) {
      if (st == 0) atomicOr(p.status + b, ok ? TV_DEV_CAPACITY : TV_DEV_BAD_TREE);
      p.tickets[b] = 0;
    }
    return;
  }
  if (F == 0 || n >= p.budget) {
    if (tid == 0) {
      p.level_start[b] = n;
      p.tickets[b] = 0;
    }
    return;
  }
  const int keep = request_merge(sh, p, b, n, ls, F);
  if (tid == 0) {
    p.n_nodes[b] = n + keep;
    p.level_start[b] = n;
    p.tickets[b] = 0;  // ready for the next call
  }
}

}  // namespace tv

namespace {
int expand_slices(int V) { return (V + tv::kExpSlice - 1) / tv::kExpSlice; }
size_t expand_ws_bytes(int B, int max_frontier, int V) {
  const size_t part = (size_t)B * max_frontier * expand_slices(V) * sizeof(tv::ExpPart);
  return ((part + 255) & ~size_t(255)) + (size_t)B * sizeof(int32_t);
}
}  // namespace

extern "C" size_t tv_tree_expand_workspace(int B, int max_frontier, int V) {
  if (B <= 0 || max_frontier <= 0 || V <= 0) return 0;
  return expand_ws_bytes(B, max_frontier, V);
}

extern "C" int tv_tree_expand(const float* draft_logits, int32_t* parents, int32_t* tokens, float* scores,
                              int32_t* n_nodes, int32_t* level_start, float* entropy, int32_t* width, int B,
                              int n_max, int V, int top_k, int max_new, int budget, int max_frontier, void* ws,
                              size_t ws_bytes, int32_t* status, void* stream) {
  tv::clear_error();
  TV_REQUIRE(draft_logits && parents && tokens && scores && n_nodes && level_start && status, TV_ERR_INVALID_ARG,
             "tv_tree_expand: NULL pointer");
  TV_REQUIRE(B >= 0 && V >= 1, TV_ERR_INVALID_ARG, "tv_tree_expand: bad sizes B=%d V=%d", B, V);
  TV_REQUIRE(n_max >= 1 && n_max <= tv::kMaxNodes, TV_ERR_UNSUPPORTED, "tv_tree_expand: n_max = %d not in [1, 64]",
             n_max);
  TV_REQUIRE(top_k >= 1 && top_k <= tv::kExpTop, TV_ERR_UNSUPPORTED, "tv_tree_expand: top_k = %d not in [1, 8]",
             top_k);
  TV_REQUIRE(max_new >= 1 && budget >= 1 && budget <= n_max, TV_ERR_INVALID_ARG,
             "tv_tree_expand: max_new = %d, budget = %d (need max_new >= 1, 1 <= budget <= n_max)", max_new, budget);
  TV_REQUIRE(max_frontier >= 1 && max_frontier <= n_max, TV_ERR_INVALID_ARG,
             "tv_tree_expand: max_frontier = %d not in [1, n_max]", max_frontier);
  TV_REQUIRE(tv::aligned16(draft_logits), TV_ERR_INVALID_ARG, "tv_tree_expand: logits must be 16-byte aligned");
  TV_REQUIRE(B <= 65535, TV_ERR_UNSUPPORTED, "tv_tree_expand: B = %d above 65535", B);
  if (B == 0) return TV_OK;
  const size_t need = expand_ws_bytes(B, max_frontier, V);
  TV_REQUIRE(ws != nullptr && ws_bytes >= need && tv::aligned16(ws), TV_ERR_WORKSPACE,
             "tv_tree_expand: workspace of %zu bytes (16-byte aligned, zero-filled once) required, got %zu", need,
             ws ? ws_bytes : (size_t)0);
  tv::ExpandParams q;
  q.logits = draft_logits;
  q.parents = parents;
  q.tokens = tokens;
  q.scores = scores;
  q.n_nodes = n_nodes;
  q.level_start = level_start;
  q.entropy = entropy;
  q.width = width;
  q.n_max = n_max;
  q.V = V;
  q.top_k = top_k;
  q.max_new = max_new;
  q.budget = budget;
  q.max_frontier = max_frontier;
  q.n_slices = expand_slices(V);
  q.part = reinterpret_cast<tv::ExpPart*>(ws);
  q.tickets = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + (need - (size_t)B * sizeof(int32_t)));
  q.status = status;
  for (int j = 0; j < tv::kExpTop; ++j) q.width_ln[j] = (float)std::log((double)j + 0.5);
  TV_CUDA_CHECK(tv::launch_pdl(tv::tree_expand_kernel, dim3(q.n_slices, max_frontier, B), dim3(tv::kExpThreads), 0,
                               tv::as_stream(stream), q));
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
}
