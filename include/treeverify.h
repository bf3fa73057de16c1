/*
 * treeverify.h — C ABI of the GB300 (sm_103a) tree-verification library
 * (libtreeverify.so).
 *
 * The library implements the target model's verification step of EAGLE-style
 * speculative decoding: a draft tree of at most 64 nodes (a parent-index
 * array, node 0 = root) is scored by one tree-masked attention pass over each
 * request's paged KV cache; the longest accepted root-to-node path is found
 * (greedy argmax match, or rejection sampling with residual resampling at
 * temperature T); the accepted branch's K/V is compacted into contiguous
 * cache slots and the rejected branches are dropped.
 *
 * Sources (three pages on EAGLE speculative decoding):
 *  - "SGLang EAGLE-2 Speculative Decoding" (Tech Radar), section 2,
 *    "Dynamic Tree-Attention Masking": tree of <= 64 candidates, mask
 *    M[i][j] = 1 iff j is an ancestor of i or i itself; one forward pass over
 *    the whole tree; the sequence diagram of the same section: keep the KV of
 *    the accepted branch, drop the wrong branches, return the verified tokens.
 *  - troisinh.com "EAGLE — Draft head ...", "Why it works": verification is
 *    rejection sampling and is lossless.
 *  - study note "EAGLE" (estelledc.github.io), case 1 (k hits emit k+1
 *    tokens) and case 3 (reject by the difference probability, resample).
 *
 * Conventions shared by every call
 *  - Every pointer argument is a DEVICE pointer owned by the caller, except
 *    where stated.  The library never allocates device memory, keeps no state
 *    across calls other than cached kernel attributes, and never synchronises
 *    the stream; all work is enqueued on `stream` (a cudaStream_t passed as
 *    void*; NULL = the legacy default stream).
 *  - B = number of requests, n_max = row stride of the per-node arrays
 *    (1 <= n_nodes[b] <= n_max <= 64).  Hq / Hkv = query / KV heads,
 *    G = Hq / Hkv query heads share KV head h / G.  D = head dim (64 or 128).
 *    page_size must be 16.
 *  - Host-side argument errors return a negative TV_ERR_* code before any
 *    launch.  Data errors found on the device never trap: they are OR-ed into
 *    the per-request int32 `status` word as TV_DEV_* bits and that request's
 *    outputs are written as documented (zeros / -1).  tv_tree_build_mask
 *    writes `status`; the other calls read it as the calls before them left
 *    it, treat requests whose status is non-zero as skipped (the documented
 *    outputs of a skipped request) and OR in their own bits.
 *  - Return value: TV_OK (0) or a negative TV_ERR_* code; tv_last_error()
 *    gives a message for the calling thread's last failure.
 *  - Launch order: every kernel is launched with programmatic dependent
 *    launch and waits for the preceding kernel in the stream before it writes
 *    any output, and before it reads anything that a call of this library
 *    writes (status, masks, accept outputs, caches).  Two calls read some of
 *    their inputs before that wait: tv_tree_accept its logits, tokens,
 *    parents, n_nodes and uniforms (and fills its own workspace), and
 *    tv_tree_verify_attn(_q4/_q3) its prefix_len, n_nodes, q, page table and
 *    K/V cache (to plan its work and load its first tiles).  Only
 *    tv_tree_build_mask and tv_tree_verify_attn(_q4/_q3) let the next kernel
 *    in the stream be scheduled before they finish, and neither writes those
 *    inputs; the calls that may write them (tv_tree_expand: parents, tokens,
 *    n_nodes; tv_kv_commit_path: the cache, and new_len, which a caller may
 *    pass as next step's prefix_len; tv_kv_prune_pages: the page table;
 *    tv_kv_quantize_q4/_q3: the low-bit cache) start their successor only
 *    after they finish.  So a kernel of the caller's that is launched with the
 *    programmatic-launch attribute must wait (griddepcontrol.wait /
 *    cudaGridDependencySynchronize) before reading the outputs of a call it
 *    follows, and one that precedes tv_tree_accept or the attention and
 *    signals its dependents early must have written those inputs before it
 *    signals.  Kernels launched without that attribute, and host
 *    synchronisation, are unaffected.
 */
#ifndef TREEVERIFY_H_
#define TREEVERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* host return codes */
#define TV_OK                0
#define TV_ERR_INVALID_ARG  (-1)  /* NULL pointer, bad size, misaligned pointer          */
#define TV_ERR_UNSUPPORTED  (-2)  /* D not in {64,128}, page_size != 16, Hq % Hkv != 0 ... */
#define TV_ERR_WORKSPACE    (-3)  /* workspace smaller than the *_workspace() query        */
#define TV_ERR_CUDA         (-4)  /* a CUDA runtime call or launch failed                  */

/* tv_tree_accept flags */
#define TV_ACCEPT_SIBLINGS_WITHOUT_REPLACEMENT 1  /* renormalise q without each rejected sibling's token */

/* device status bits (per request, OR-ed) */
#define TV_DEV_BAD_TREE   1   /* parent[0] != -1, parent[i] not in [0, i), n_nodes not in [1, n_max] */
#define TV_DEV_PAGE_OOB   2   /* a needed page id is outside [0, num_pages)                        */
#define TV_DEV_CAPACITY   4   /* L + N positions do not fit in max_pages * page_size               */
#define TV_DEV_TIMEOUT    8   /* a bounded on-chip wait gave up (about one second)                */
#define TV_DEV_BAD_TOKEN 16   /* a drafted token id is outside [0, V)                              */
#define TV_DEV_BAD_REFCOUNT 32 /* a page released by tv_kv_prune_pages had a reference count of 0    */

/*
 * Workspace size in bytes that tv_tree_expand needs for B requests, frontiers
 * of at most max_frontier nodes and vocabulary V: per-slice partials of every
 * frontier row (80 bytes per 8192-logit slice) plus one arrival counter per
 * request.  The workspace (16-byte aligned) must be zero-filled before its
 * first use; every call leaves the counters at zero again, so one workspace
 * serves any number of calls issued in order on one stream.
 */
size_t tv_tree_expand_workspace(int B, int max_frontier, int V);

/*
 * tv_tree_expand — one level of dynamic draft-tree construction, the drafting
 * loop that builds the tree the other calls verify ("SGLang EAGLE-2
 * Speculative Decoding" (Tech Radar), section 2: per expansion depth the
 * drafter's distribution is scored by its entropy H = -sum P log P, natural
 * log ("Dynamic Tree-Attention Masking"); low entropy extends one branch,
 * high entropy widens the tree up to 8 children; beam search prunes the low
 * branches (sequence diagram); the tree holds at most 64 nodes).
 *
 * State per request b (updated in place): nodes [0, n_nodes[b]) with parents,
 * tokens and cumulative log-probabilities `scores`; the frontier is the last
 * level added, nodes [level_start[b], n_nodes[b]).  Start a tree with
 * n_nodes = 1, level_start = 0, parents[0] = -1, tokens[0] = the last verified
 * token, scores[0] = 0, then call once per depth (4-6 in the pages).
 *
 * For each frontier node f: P = softmax(draft_logits[b][f]);
 * w_f = round(e^H) clamped to [1, top_k] (H at or above ln(j + 1/2) gives more
 * than j children); candidates are f's w_f most probable tokens (equal logits:
 * lower token id first) with score scores[f] + log P(token).  The best
 * keep = min(max_new, budget - n_nodes[b], candidates) by score (equal scores:
 * lower f, then lower rank) become nodes n_nodes[b] .. n_nodes[b] + keep - 1,
 * in (f, rank) order: parents precede children, siblings are contiguous, most
 * probable first.  Then level_start[b] = old n_nodes[b] and n_nodes[b] += keep
 * (keep = 0 leaves an empty frontier).  Entries past the old n_nodes[b] are
 * written only up to the new n_nodes[b].
 *
 *  draft_logits float [B, n_max, V]  row f = the drafter's logits for the
 *    children of node f (finite values; only frontier rows are read).  The
 *    same rows are the q rows tv_tree_accept takes when sampling.
 *  parents, tokens  int32 [B, n_max]  in/out
 *  scores   float [B, n_max]  in/out, cumulative natural-log probability
 *  n_nodes, level_start  int32 [B]  in/out
 *  entropy  float [B, n_max]  out (may be NULL): H of each frontier row
 *  width    int32 [B, n_max]  out (may be NULL): w_f of each frontier row
 *  top_k    1..8 (largest branching); max_new >= 1 (nodes one level may add);
 *  budget   1..n_max (node cap of the tree); max_frontier 1..n_max: an upper
 *    bound on every request's frontier (max_new, or 1 for the first level)
 *  ws, ws_bytes  workspace of at least tv_tree_expand_workspace(B,
 *    max_frontier, V) bytes
 *  status   int32 [B]  in/out: requests with non-zero status are skipped;
 *    an invalid state (n_nodes not in [1, n_max] or level_start not in
 *    [0, n_nodes]) ORs TV_DEV_BAD_TREE and a frontier larger than
 *    max_frontier ORs TV_DEV_CAPACITY; the state is then left unchanged.
 */
int tv_tree_expand(const float* draft_logits, int32_t* parents, int32_t* tokens, float* scores, int32_t* n_nodes,
                   int32_t* level_start, float* entropy, int32_t* width, int B, int n_max, int V, int top_k,
                   int max_new, int budget, int max_frontier, void* ws, size_t ws_bytes, int32_t* status,
                   void* stream);

/*
 * tv_tree_build_mask — the tree-attention mask (Tech Radar section 2, the mask
 * M: bit j of anc_mask[b][i] is set iff node j is an ancestor of node i or i
 * itself) and each node's depth (root = 0; RoPE positions are L + depth).
 *
 *  parents  int32 [B, n_max]  parent index per node, parents[b][0] = -1
 *  n_nodes  int32 [B]         nodes of request b
 *  anc_mask uint64 [B, n_max] out; entries i >= n_nodes[b] are 0
 *  depth    int32 [B, n_max]  out; entries i >= n_nodes[b] are -1
 *  status   int32 [B]         out (written, not OR-ed): 0 or TV_DEV_BAD_TREE
 *                             (an invalid tree gets all-zero mask / -1 depth)
 */
int tv_tree_build_mask(const int32_t* parents, const int32_t* n_nodes, int B, int n_max,
                       uint64_t* anc_mask, int32_t* depth, int32_t* status, void* stream);

/*
 * Workspace size in bytes that tv_tree_verify_attn needs for these sizes
 * (split-KV partial outputs, split tickets, error bits, an exit counter).
 * The caller zero-fills the workspace once after allocating it; every call
 * leaves it zeroed again, so it can be reused by later calls of the same
 * sizes.  Calls that may overlap in time need separate workspaces.
 * max_kv_len is accepted for interface stability and is not used.
 */
size_t tv_tree_verify_attn_workspace(int B, int n_max, int Hq, int Hkv, int D, int max_kv_len);

/*
 * tv_tree_verify_attn — one tree-masked attention pass of every tree node over
 * its request's paged KV cache (Tech Radar section 2: one forward pass scores
 * every branch, with the mask M).  For request b, query head h, node i:
 *
 *   visible keys = prefix positions 0..L-1  and  tree positions L+j, j in A(i)
 *   s_t = scale * <q, k_t>,  out = sum_t softmax(s)_t v_t,
 *   lse = ln sum_t exp(s_t)
 *
 * where L = prefix_len[b] and A(i) = ancestors of i plus i (anc_mask[b][i]).
 * Bits j >= n_nodes[b] of a node's word are ignored (only the request's own
 * tree positions L..L+N-1 can be made visible).
 * The tree's own K/V must already sit at logical positions L..L+N-1 of the
 * request's pages; logical position t lives in physical page
 * page_table[b][t / 16], row t % 16.
 *
 *  q          bf16 [B, n_max, Hq, D]          (16-byte aligned)
 *  k_cache    bf16 [num_pages, Hkv, 16, D]     (16-byte aligned)
 *  v_cache    bf16 [num_pages, Hkv, 16, D]     (16-byte aligned)
 *  page_table int32 [B, max_pages]
 *  prefix_len int32 [B], n_nodes int32 [B], anc_mask uint64 [B, n_max]
 *  out        bf16 [B, n_max, Hq, D]  out; rows i >= n_nodes[b] untouched; a
 *                                      request with non-zero status gets zeros in
 *                                      all n_max rows (and in lse)
 *  lse        float [B, n_max, Hq]    out, may be NULL
 *  ws/ws_bytes  device workspace of at least tv_tree_verify_attn_workspace() bytes
 *  status     int32 [B]  in/out: TV_DEV_PAGE_OOB | TV_DEV_CAPACITY | TV_DEV_TIMEOUT
 *
 * Returns TV_ERR_UNSUPPORTED for D not in {64,128}, page_size != 16,
 * Hq % Hkv != 0, 128 % G != 0 or B > 1024.  One kernel launch: the work is
 * divided evenly over the SMs and split key ranges are merged in-kernel.
 */
int tv_tree_verify_attn(const void* q, const void* k_cache, const void* v_cache, int64_t num_pages,
                        const int32_t* page_table, int max_pages, const int32_t* prefix_len,
                        const int32_t* n_nodes, const uint64_t* anc_mask, int B, int n_max, int Hq,
                        int Hkv, int D, int page_size, float scale, void* out, float* lse, void* ws,
                        size_t ws_bytes, int32_t* status, void* stream);

/*
 * tv_tree_verify_attn_noalloc — the same computation as tv_tree_verify_attn
 * (same arguments, outputs and status behaviour) without a caller workspace.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory on their own — for example code embedded in a
 * host framework that owns every device allocation, or plug-ins that may only
 * touch the buffers they are handed.  Its scratch is a fixed 48 MiB array
 * compiled into the library; every device that loads the library holds it
 * until the process exits.
 *  - The first call on each device looks up the array's device address (with
 *    that device current) and caches it together with the id of the current
 *    context; make that first call before any stream capture.  A call in a new
 *    context on the device (after cudaDeviceReset, say) looks the address up
 *    again, so that first call after a reset should also precede any capture.
 *  - The scratch need is 2 * SMs * 256 * (2 * D + 8) bytes of split partials
 *    plus 8 bytes per (request, KV head, M-tile pair) of split tickets: about
 *    20.6 MB at D = 128 on 152 SMs for every workload shape this library is
 *    measured on (the largest ticket area among them is 4 KB), well inside
 *    48 MiB.
 *  - Sizes whose scratch need exceeds 48 MiB return TV_ERR_UNSUPPORTED with a
 *    message; use tv_tree_verify_attn with a workspace for those.
 *  - Every call shares the one array and clears its counters at the start
 *    (an asynchronous memset on `stream`), so calls that may overlap on the
 *    GPU (other streams, other threads) race and must be serialised by the
 *    caller.
 *  - The call itself allocates nothing.
 */
int tv_tree_verify_attn_noalloc(const void* q, const void* k_cache, const void* v_cache, int64_t num_pages,
                                const int32_t* page_table, int max_pages, const int32_t* prefix_len,
                                const int32_t* n_nodes, const uint64_t* anc_mask, int B, int n_max, int Hq,
                                int Hkv, int D, int page_size, float scale, void* out, float* lse,
                                int32_t* status, void* stream);

/*
 * Workspace size in bytes that tv_tree_accept needs for these sizes.  It is
 * non-zero when B * n_max * V * 4 <= 64 MiB: there a greedy call reads every
 * node's logits in one parallel pass (per-slice partial argmaxes plus one
 * arrival counter per request) instead of one dependent row read per tree
 * level.  The workspace (16-byte aligned) must be zero-filled before its first
 * use; every call leaves the counters at zero again, so one workspace serves
 * any number of calls issued in order on one stream.  0: none needed.
 */
size_t tv_tree_accept_workspace(int B, int n_max, int V);

/*
 * tv_tree_accept — find the longest accepted root-to-node path and the tokens
 * to emit.
 *
 * Greedy (temperature == 0): node j (non-root) hits iff tokens[j] equals the
 * argmax of target_logits at parent(j) (lowest index on ties); node c is
 * accepted iff every non-root node on its root path hits; the result is the
 * deepest accepted node (lowest index on ties); the bonus token is the argmax
 * at the result (k hits emit k+1 tokens: study note case 1).
 *
 * Sampling (temperature > 0): walk from the root; at node n let
 * p = softmax(target[n]/T), q = softmax(draft[n]/T); try n's children c in
 * ascending index: accept iff u_accept[c] * q(x_c) < p(x_c); on rejection
 * replace p by max(0, p - q) normalised (unchanged if that sums to 0).  The
 * first accepted child becomes the next node.  When no child is accepted (or n
 * is a leaf) the bonus token is min{ j : u_sample[n] * S < C_j } over the
 * running sum C of the current p (troisinh.com "Why it works"; study note
 * case 3).
 *
 * TV_ACCEPT_SIBLINGS_WITHOUT_REPLACEMENT: for trees whose siblings were drafted
 * without replacement (distinct tokens, e.g. Gumbel top-k): after child c with
 * token x is rejected, q also loses x and is renormalised before the next
 * sibling (q(x) <- 0, q <- q / sum q; all zero when nothing is left); the
 * residual step itself uses the q that c was tested against.  Sequential
 * rejection against the renormalised draft keeps the output distribution
 * exactly the target's under such drafting, as the fixed-q rule does under
 * i.i.d. drafting.
 * Which rule is lossless depends only on how the children were drafted: a tree
 * grown by sampled top-k expansion (distinct sibling tokens, e.g. the Gumbel
 * top-k of the draft row) needs this flag; children drawn independently from
 * q (repeats allowed) need flags = 0.  Neither rule is lossless for the
 * other's drafting, and a deterministic top-k (argmax) expansion is lossless
 * under neither.
 *
 *  target_logits float [B, n_max, V]; draft_logits float [B, n_max, V] (row n =
 *    the distribution n's children were drawn from; may be NULL when greedy)
 *  tokens   int32 [B, n_max]  drafted token of each node (root entry ignored)
 *  parents, n_nodes, anc_mask, depth: as produced by tv_tree_build_mask
 *  flags    0, or TV_ACCEPT_SIBLINGS_WITHOUT_REPLACEMENT (sampling only; see below)
 *  u_accept, u_sample  float [B, n_max] uniforms in [0, 1) (unused when greedy)
 *  accept_len  int32 [B]          out: accepted non-root nodes a
 *  path_nodes  int32 [B, n_max]   out: 0, n_1 .. n_a, then -1
 *  out_tokens  int32 [B, n_max+1] out: tokens of n_1..n_a, the bonus, then -1
 *  ws, ws_bytes  workspace of at least tv_tree_accept_workspace(B, n_max, V)
 *                bytes (may be NULL when that is 0); TV_ERR_INVALID_ARG if smaller
 *  status      int32 [B]          in/out: TV_DEV_BAD_TOKEN, TV_DEV_TIMEOUT
 *
 * Sampling holds each request's two rows in registers across one cluster of
 * at most 16 CTAs: V <= 262144 (TV_ERR_UNSUPPORTED above).  Greedy has no
 * limit on V.
 */
int tv_tree_accept(const float* target_logits, const float* draft_logits, const int32_t* tokens,
                   const int32_t* parents, const int32_t* n_nodes, const uint64_t* anc_mask,
                   const int32_t* depth, int B, int n_max, int V, float temperature, int flags,
                   const float* u_accept, const float* u_sample, int32_t* accept_len,
                   int32_t* path_nodes, int32_t* out_tokens, void* ws, size_t ws_bytes,
                   int32_t* status, void* stream);

/*
 * tv_kv_commit_path — keep the accepted branch's K/V, drop the rejected ones
 * (Tech Radar section 2, sequence diagram).  For k = 1..a (a = accept_len[b],
 * n_k = path_nodes[b][k]) the K and V rows at logical position L + n_k move
 * to L + k, in every layer and KV head; the root stays at L.  Moves with
 * n_k == k are skipped; a source is always read before any overlapping
 * destination is written.
 *
 *  k_cache, v_cache   bf16; layer l's cache [num_pages, Hkv, 16, D] starts
 *                     layer_stride_elems elements after layer l-1's (16-byte aligned)
 *  committed_slots    int64 [B, n_max] out: page_table[(L+k)/16]*16 + (L+k)%16
 *                     for k = 0..a, then -1
 *  new_len            int32 [B] out: L + a + 1 (L for a request with non-zero status)
 *  status             int32 [B] in/out: TV_DEV_PAGE_OOB | TV_DEV_CAPACITY | TV_DEV_BAD_TREE
 *                     (a path that is not a root-first increasing chain)
 */
int tv_kv_commit_path(void* k_cache, void* v_cache, int n_layers, int64_t layer_stride_elems,
                      int64_t num_pages, const int32_t* page_table, int max_pages,
                      const int32_t* prefix_len, const int32_t* n_nodes, const int32_t* accept_len,
                      const int32_t* path_nodes, int B, int n_max, int Hkv, int D, int page_size,
                      int64_t* committed_slots, int32_t* new_len, int32_t* status, void* stream);

/*
 * tv_kv_prune_pages — release, without copying, the pages that hold only
 * rejected tree rows once the accepted path has been committed ("SGLang
 * EAGLE-2 Speculative Decoding" (Tech Radar), failure mode 2: rejected
 * branches leave garbage blocks in the page table, and a prefix-tree page
 * manager frees them at once without a copy; section 2's sequence diagram:
 * keep the accepted branch, drop the wrong branches).
 *
 * Request b keeps positions [0, new_len[b]) (new_len from tv_kv_commit_path).
 * Page-table slots ceil(new_len / 16) .. ceil((L + N) / 16) - 1 hold no kept
 * position: each is set to -1 and refcount[page] drops by one; a page whose
 * count reaches 0 is appended to free_list (at index *free_count, which is
 * advanced; the order of pages freed by one call is unspecified).  Pages whose
 * count stays above 0 (shared with other sequences, e.g. a radix-tree prefix)
 * remain in use.  Nothing else is read or written; no K/V row moves.
 *
 *  page_table  int32 [B, max_pages]  in/out
 *  refcount    int32 [num_pages]     in/out, references held on each page
 *  prefix_len, n_nodes, new_len  int32 [B]  (L, N, and L + accept_len + 1)
 *  page_size   must be 16
 *  free_list   int32 [free_capacity] out (may be NULL when free_capacity = 0)
 *  free_count  int32 [1]             in/out
 *  status      int32 [B] in/out: requests with non-zero status are skipped;
 *    TV_DEV_CAPACITY when L + N does not fit the row (or L < 0) or when the
 *    free list is full (the page is then free but not listed); TV_DEV_BAD_TREE
 *    when new_len is not in [L + 1, L + N]; TV_DEV_PAGE_OOB when a released
 *    slot holds an id outside [0, num_pages) (nothing released);
 *    TV_DEV_BAD_REFCOUNT when a released page's count is already 0 (the slot
 *    is cleared, the count stays 0).
 * Requests may share pages: counts change atomically.
 */
int tv_kv_prune_pages(int32_t* page_table, int max_pages, int32_t* refcount, int64_t num_pages,
                      const int32_t* prefix_len, const int32_t* n_nodes, const int32_t* new_len, int B,
                      int page_size, int32_t* free_list, int64_t free_capacity, int32_t* free_count,
                      int32_t* status, void* stream);

/*
 * tv_kv_quantize_q4 — encode bf16 KV rows in a 4-bit cache format
 * (troisinh.com "EAGLE - Draft head ...": EAGLE pairs with an INT4 KV cache;
 * further reading: KV-cache quantisation to INT4/INT3).  Per row and group
 * of 32 dims: scale and zero in fp16, codes 0..15 two per byte (low nibble =
 * even dim); a value decodes to bf16(fp32(code * scale + zero)).  Encoding, in
 * fp32 with round-to-nearest-even at each step: zero = fp16(min x),
 * scale = fp16((max x - min x) / 15), inv = fp32(1 / scale),
 * code = clamp(rint((x - zero) * inv), 0, 15), or 0 when scale is 0.
 * Inputs must be finite.
 *
 *  x       bf16 [rows, D] (any row layout: a paged cache [pages, Hkv, 16, D]
 *          is pages * Hkv * 16 rows), 16-byte aligned
 *  D       a multiple of 32, at most 1024
 *  codes   uint8 [rows, D / 2] out, 16-byte aligned
 *  params  fp16 [rows, 2 * D / 32] out: (scale, zero) per group, 4-byte aligned
 */
int tv_kv_quantize_q4(const void* x, int64_t rows, int D, uint8_t* codes, void* params, void* stream);

/*
 * tv_tree_verify_attn_q4 — tv_tree_verify_attn over a paged KV cache held in
 * the 4-bit format of tv_kv_quantize_q4 (troisinh.com "EAGLE - Draft head
 * ...": EAGLE pairs with an INT4 KV cache).  The result is that of
 * tv_tree_verify_attn on the decoded cache: every K and V value is first
 * decoded to bf16(fp32(code * scale + zero)) with its row's (scale, zero) of
 * its 32-dim group; the kernel decodes each page in shared memory as it
 * streams, and the cache is read at about 0.31 (D = 128) of the bf16 bytes.
 *
 *  q          bf16 [B, n_max, Hq, D]                    (16-byte aligned)
 *  k_codes    uint8 [num_pages, Hkv, 16, D / 2]         (16-byte aligned)
 *  k_params   fp16  [num_pages, Hkv, 16, 2 * D / 32]    (16-byte aligned)
 *  v_codes, v_params  the same for V
 *  every other argument, the outputs, the workspace (tv_tree_verify_attn_workspace
 *  of the same sizes) and the status bits as for tv_tree_verify_attn.
 *
 * Returns TV_ERR_UNSUPPORTED for D not in {64,128}, page_size != 16,
 * Hq % Hkv != 0, 128 % G != 0 or B > 256.  One kernel launch.
 */
int tv_tree_verify_attn_q4(const void* q, const uint8_t* k_codes, const void* k_params, const uint8_t* v_codes,
                           const void* v_params, int64_t num_pages, const int32_t* page_table, int max_pages,
                           const int32_t* prefix_len, const int32_t* n_nodes, const uint64_t* anc_mask, int B,
                           int n_max, int Hq, int Hkv, int D, int page_size, float scale, void* out, float* lse,
                           void* ws, size_t ws_bytes, int32_t* status, void* stream);

/*
 * tv_kv_quantize_q3 — encode bf16 KV rows in a 3-bit cache format
 * (troisinh.com "EAGLE - Draft head ...", further reading: KV-cache
 * quantisation to INT4/INT3).  Per row and group of 32 dims: scale and zero
 * in fp16 as for tv_kv_quantize_q4, codes 0..7.  A row's codes take 3 * D / 8
 * bytes: first the low two bits of every code, four per byte (byte j: dims
 * 4j .. 4j+3, dim 4j+i in bits 2i and 2i+1), then the third bits, eight per
 * byte (byte D/4 + j: dims 8j .. 8j+7, dim 8j+i in bit i).  A value decodes to
 * bf16(fp32(code * scale + zero)).  Encoding, in fp32 with round-to-nearest-
 * even at each step: zero = fp16(min x), scale = fp16((max x - min x) / 7),
 * inv = fp32(1 / scale), code = clamp(rint((x - zero) * inv), 0, 7), or 0 when
 * scale is 0.  Inputs must be finite.
 *
 *  x       bf16 [rows, D] (any row layout), 16-byte aligned
 *  D       a multiple of 32, at most 1024
 *  codes   uint8 [rows, 3 * D / 8] out, 4-byte aligned
 *  params  fp16 [rows, 2 * D / 32] out: (scale, zero) per group, 4-byte aligned
 */
int tv_kv_quantize_q3(const void* x, int64_t rows, int D, uint8_t* codes, void* params, void* stream);

/*
 * tv_tree_verify_attn_q3 — tv_tree_verify_attn over a paged KV cache held in
 * the 3-bit format of tv_kv_quantize_q3: the result is that of
 * tv_tree_verify_attn on the decoded cache (every K and V value first decoded
 * to bf16(fp32(code * scale + zero))); the kernel decodes each page in shared
 * memory as it streams, reading the cache at about 0.25 (D = 128) of the bf16
 * bytes.
 *
 *  q          bf16 [B, n_max, Hq, D]                    (16-byte aligned)
 *  k_codes    uint8 [num_pages, Hkv, 16, 3 * D / 8]     (16-byte aligned)
 *  k_params   fp16  [num_pages, Hkv, 16, 2 * D / 32]    (16-byte aligned)
 *  v_codes, v_params  the same for V
 *  everything else as for tv_tree_verify_attn_q4.
 */
int tv_tree_verify_attn_q3(const void* q, const uint8_t* k_codes, const void* k_params, const uint8_t* v_codes,
                           const void* v_params, int64_t num_pages, const int32_t* page_table, int max_pages,
                           const int32_t* prefix_len, const int32_t* n_nodes, const uint64_t* anc_mask, int B,
                           int n_max, int Hq, int Hkv, int D, int page_size, float scale, void* out, float* lse,
                           void* ws, size_t ws_bytes, int32_t* status, void* stream);

/*
 * tv_selftest_wait_timeout — self-test of the bounded waits every kernel uses
 * (no counterpart in the pages).  One CTA waits on an mbarrier that nothing
 * ever completes; after the wait limit (1 s) it ORs TV_DEV_TIMEOUT into
 * *status (int32, device) and returns.  Nothing traps and the context stays
 * usable.  Asynchronous on `stream`; expect about one second of GPU time.
 */
int tv_selftest_wait_timeout(int32_t* status, void* stream);

/* Message for the calling thread's last failed call ("" if none). */
const char* tv_last_error(void);

/* Library version string. */
const char* tv_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TREEVERIFY_H_ */
