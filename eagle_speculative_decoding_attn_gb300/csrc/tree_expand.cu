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
  ExpPart* part;      // [B][max_frontier][n_slices]
  int32_t* tickets;   // [B] arrivals of this call (zero between calls)
  int32_t* status;
};

struct ExpShared {
  float red_m[kExpWarps], red_s[kExpWarps], red_t[kExpWarps], wmax[kExpWarps];
  float wtop_v[kExpWarps][kExpTop];
  int wtop_i[kExpWarps][kExpTop];
  float top_v[kExpTop];
  int top_i[kExpTop];
  float cand_v[kSliceCand];
  int cand_i[kSliceCand];
  int cand_n;
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

// Reduce one slice (x in registers) to its part and store it at dst (thread 0
// writes it; it publishes the part with a fence before arriving).
__device__ __forceinline__ void slice_reduce(ExpShared& sh, const float (&x)[kExpPerThread], bool work, int lo,
                                             int hi, ExpPart* dst) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float m = -INFINITY, s = 0.f, t = 0.f;
  if (work) {
    // four independent chains for the maximum and the two sums
    float m4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
    for (int k = 4; k < kExpPerThread; ++k) m4[k & 3] = fmaxf(m4[k & 3], x[k]);
    m = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
    float s4[4] = {0.f, 0.f, 0.f, 0.f}, t4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kExpPerThread; ++k) {
      // d >= -200 keeps e * d finite: e is then 0 (also when the thread saw
      // no logit and m = -inf, where x - m is NaN and fmaxf takes -200)
      const float d = fmaxf(x[k] - m, -200.f);
      const float e = ex2_approx(d * kLog2e);
      s4[k & 3] += e;
      t4[k & 3] = fmaf(e, d, t4[k & 3]);
    }
    s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
    t = (t4[0] + t4[1]) + (t4[2] + t4[3]);
    if (s == 0.f) m = -INFINITY;
  }
  // Each warp's largest logit is a distinct logit, so with 8 warps the
  // slice's 8 best are all >= tau, the smallest warp maximum: only logits
  // >= tau are candidates (a warp without logits makes tau = -inf).  After
  // the warp's (m, s, t) merge, m is that maximum.
  warp_mst(m, s, t);
  if (lane == 0) {
    sh.red_m[warp] = m;
    sh.red_s[warp] = s;
    sh.red_t[warp] = t;
    sh.wmax[warp] = m;
  }
  if (tid == 0) {  // the thread that reads the previous slice's list
#pragma unroll
    for (int k = 0; k < kExpTop; ++k) {
      sh.top_v[k] = -INFINITY;
      sh.top_i[k] = INT_MAX;
    }
  }
  __syncthreads();
  if (warp == 0) {  // the slice's (m, s, t)
    m = lane < kExpWarps ? sh.red_m[lane] : -INFINITY;
    s = lane < kExpWarps ? sh.red_s[lane] : 0.f;
    t = lane < kExpWarps ? sh.red_t[lane] : 0.f;
    warp_mst(m, s, t);
  }
  float tau = INFINITY;
#pragma unroll
  for (int w = 0; w < kExpWarps; ++w) tau = fminf(tau, sh.wmax[w]);
  if (work) {
#pragma unroll
    for (int u = 0; u < kExpPerThread / 4; ++u)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int j = slice_j(lo, u, c);
        if (j < hi && x[4 * u + c] >= tau) {
          const int slot = atomicAdd(&sh.cand_n, 1);
          if (slot < kSliceCand) {
            sh.cand_v[slot] = x[4 * u + c];
            sh.cand_i[slot] = j;
          }
        }
      }
  }
  __syncthreads();
  const int nc = sh.cand_n;
  if (nc <= kSliceCand) {
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
    // many logits equal to tau: exact per-thread lists instead
    float tv_[kExpTop], ov[kExpTop];
    int ti_[kExpTop], oi[kExpTop];
    top_clear(tv_, ti_);
    if (work) {
#pragma unroll
      for (int u = 0; u < kExpPerThread / 4; ++u)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int j = slice_j(lo, u, c);
          if (j < hi) top_insert(tv_, ti_, x[4 * u + c], j);
        }
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
    if (lane == 0) {
      ExpPart r;
      r.m = m;
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
  } else if (tid == 32) {
    sh.cand_n = 0;  // every thread has read it; the next slice appends after its first barrier
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
  // warp w takes rows w, w + 8, ...
  for (int r = warp; r < F; r += kExpWarps) {
    float m = -INFINITY, s = 0.f, t = 0.f;
    top_clear(tv_, ti_);
    const ExpPart* src = p.part + ((int64_t)b * p.max_frontier + r) * p.n_slices;
    for (int q = lane; q < p.n_slices; q += 32) {
      const float4* w4 = reinterpret_cast<const float4*>(src + q);
      float4 w[5];
#pragma unroll
      for (int k = 0; k < 5; ++k) w[k] = __ldcg(w4 + k);
      mst_merge(m, s, t, w[0].x, w[0].y, w[0].z);
      const float pv[kExpTop] = {w[1].x, w[1].y, w[1].z, w[1].w, w[2].x, w[2].y, w[2].z, w[2].w};
      const int pi[kExpTop] = {__float_as_int(w[3].x), __float_as_int(w[3].y), __float_as_int(w[3].z),
                               __float_as_int(w[3].w), __float_as_int(w[4].x), __float_as_int(w[4].y),
                               __float_as_int(w[4].z), __float_as_int(w[4].w)};
      if (q == lane) {  // the lane's first part: its sorted list as is
#pragma unroll
        for (int k = 0; k < kExpTop; ++k) {
          tv_[k] = pv[k];
          ti_[k] = pi[k];
        }
      } else {
#pragma unroll
        for (int k = 0; k < kExpTop; ++k)
          if (!top_insert(tv_, ti_, pv[k], pi[k])) break;  // the part's list is sorted
      }
    }
    warp_mst(m, s, t);
    warp_top8(tv_, ti_, ov, oi);
    if (lane == 0) {
      const int f = ls + r;
      const float lz = logf(s);  // log of the normaliser, relative to m
      const float H = lz - t / s;
      int w = 1;
      for (int j = 1; j < p.top_k; ++j)
        if (H >= logf((float)j + 0.5f)) w = j + 1;
      int real = 0;
#pragma unroll
      for (int k = 0; k < kExpTop; ++k) real += oi[k] != INT_MAX;
      w = min(w, real);
      if (p.entropy) p.entropy[(int64_t)b * n_max + f] = H;
      if (p.width) p.width[(int64_t)b * n_max + f] = w;
      sh.row_w[r] = w;
      const float sf = p.scores[(int64_t)b * n_max + f];
#pragma unroll
      for (int k = 0; k < kExpTop; ++k) {
        sh.row_c[r][k] = sf + ((ov[k] - m) - lz);
        sh.row_tok[r][k] = oi[k];
      }
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
#pragma unroll
  for (int h = 0; h < 2; ++h) {
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
  griddep_wait();
  const int st = p.status[b];
  const int n = p.n_nodes[b], ls = p.level_start[b];
  const bool ok = st == 0 && n >= 1 && n <= n_max && ls >= 0 && ls <= n;
  const int F = ok ? n - ls : 0;
  const bool work = ok && y < F && F <= p.max_frontier && n < p.budget;
  if (tid == 0) sh.cand_n = 0;

  float x[kExpPerThread];
  int lo = 0, hi = 0;
  if (work) {
    const float* row = p.logits + ((int64_t)b * n_max + ls + y) * V;
    lo = sl * kExpSlice;
    hi = min(V, lo + kExpSlice);
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
  }
  ExpPart* dst = p.part + ((int64_t)b * p.max_frontier + y) * p.n_slices + sl;
  slice_reduce(sh, x, work, lo, hi, dst);
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
  TV_CUDA_CHECK(tv::launch_pdl(tv::tree_expand_kernel, dim3(q.n_slices, max_frontier, B), dim3(tv::kExpThreads), 0,
                               tv::as_stream(stream), q));
  TV_CUDA_CHECK(cudaGetLastError());
  return TV_OK;
}
