"""fp64 CPU oracle for EAGLE-style tree verification.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package's smoke check and
the benchmark's CPU-baseline / reference arm may import this module.  The
product path (the CUDA library and its binding) never calls it, and this
module imports nothing from the product package.

Each function is the plain definition of one step of the verification step,
written for readability rather than speed: explicit loops over requests,
nodes and heads, numpy fp64 arithmetic, no blocking, fusion or reordering.

Sources (the three pages on EAGLE speculative decoding):
  * "SGLang EAGLE-2 Speculative Decoding" (Tech Radar), section 2,
    "Dynamic Tree-Attention Masking": a candidate tree of at most 64 nodes is
    encoded as a mask M in {0,1}^{KxK} with M[i][j] = 1 iff j is an ancestor
    of i or i itself; one forward pass scores every branch; the target then
    keeps the KV of the accepted branch and drops the wrong ones (sequence
    diagram of the same section).
  * "EAGLE - Draft head ..." (troisinh.com), section "Why it works",
    paragraph on verification probability: verification is rejection
    sampling; a wrong draft is resampled from the correct distribution, so the
    output distribution equals plain autoregressive decoding.
  * "EAGLE" study note (estelledc.github.io), case 3: accept a candidate the
    target finds likely, otherwise reject with the difference probability and
    resample; case 1: k drafted hits advance k+1 tokens.
  * Tech Radar section 2 again for the drafting loop before verification
    (step 0): per depth (4-6) the entropy H = -sum P log P of the draft
    distribution is scored, then beam search prunes the low branches; low
    entropy extends one branch, high entropy widens up to 8 nodes.

Readings where the pages are silent (each one is listed in the design notes):
  * multi-child rule: children are tried in ascending node index with the
    draft distribution q fixed; after a rejected child the target
    distribution is replaced by the normalised residual max(0, p - q);
    for siblings drafted without replacement (distinct tokens, top-k trees)
    the selectable variant also removes each rejected token from q and
    renormalises it before the next sibling;
  * ties: argmax -> lowest vocab index; deepest accepted node -> lowest node
    index; inverse CDF -> first index j with u*S < C_j (strict);
  * temperature: softmax(z / T); T = 0 means greedy;
  * GQA: query head h reads KV head h // (Hq / Hkv);
  * scale is given by the caller (1/sqrt(D) in every workload); the
    log-sum-exp is in natural log.
  * tree expansion: a frontier node gets round(e^H) children (natural log,
    clamped to [1, top_k]); candidates are its most probable tokens scored by
    cumulative log-probability; per level the best min(max_new, budget -
    n_nodes) are kept (equal scores: lower parent, then lower rank) and
    appended in (parent, rank) order.

Every function here is pinned by tests in ``tests/test_oracle_*.py`` against
facts that do not come from this file (library routines, closed forms,
brute force, enumeration and hand-derived fixtures).
"""
from __future__ import annotations

import numpy as np

# Device status bits, restated from the library's interface definition.
STATUS_OK = 0
STATUS_BAD_TREE = 1
STATUS_PAGE_OOB = 2
STATUS_CAPACITY = 4
STATUS_TIMEOUT = 8
STATUS_BAD_TOKEN = 16
STATUS_BAD_REFCOUNT = 32

MAX_NODES = 64
NEAR_BOUNDARY = 1e-6


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode raw bf16 bit patterns (uint16) to float64 exactly."""
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def tree_is_valid(parents_row: np.ndarray, n: int) -> bool:
    """A tree is 1..64 nodes, node 0 is the root (parent -1) and every other
    node's parent precedes it."""
    if n < 1 or n > MAX_NODES:
        return False
    if int(parents_row[0]) != -1:
        return False
    for i in range(1, n):
        p = int(parents_row[i])
        if p < 0 or p >= i:
            return False
    return True


def ancestors_or_self(parents_row: np.ndarray, i: int) -> list:
    """Walk parent links from node i up to the root; returns root-first list
    [0, ..., parent(i), i]."""
    path = [i]
    while path[-1] != 0:
        path.append(int(parents_row[path[-1]]))
    return path[::-1]


# --------------------------------------------------------------------------
# step 1: tree mask
# --------------------------------------------------------------------------
def tree_build_mask(parents: np.ndarray, n_nodes: np.ndarray):
    """Ancestor mask of each node as a 64-bit word: bit j set iff node j is an
    ancestor of i or i itself (Tech Radar section 2, the mask M), plus the
    node's depth (root = 0).

    Returns (anc_mask uint64 [B, n_max], depth int32 [B, n_max], status int32 [B]).
    Entries past n_nodes[b] are 0 (mask) and -1 (depth); an invalid tree gets
    STATUS_BAD_TREE and all-zero / -1 outputs.
    """
    parents = np.asarray(parents)
    B, n_max = parents.shape
    anc = np.zeros((B, n_max), dtype=np.uint64)
    depth = np.full((B, n_max), -1, dtype=np.int32)
    status = np.zeros(B, dtype=np.int32)
    for b in range(B):
        n = int(n_nodes[b])
        if n > n_max or not tree_is_valid(parents[b], n):
            status[b] = STATUS_BAD_TREE
            continue
        for i in range(n):
            path = ancestors_or_self(parents[b], i)
            word = 0
            for j in path:
                word |= 1 << j
            anc[b, i] = np.uint64(word)
            depth[b, i] = len(path) - 1
    return anc, depth, status


# --------------------------------------------------------------------------
# step 2: tree-verify attention
# --------------------------------------------------------------------------
def _request_pages_ok(page_table_row, L, N, num_pages, page_size):
    """CAPACITY when the prefix length is negative or the L + N positions do
    not fit in the request's page-table row; otherwise PAGE_OOB when one of
    the pages holding them is outside [0, num_pages)."""
    if L < 0 or N < 1:
        return STATUS_CAPACITY
    need = (L + N + page_size - 1) // page_size
    if need > len(page_table_row):
        return STATUS_CAPACITY
    for k in range(need):
        if not (0 <= int(page_table_row[k]) < num_pages):
            return STATUS_PAGE_OOB
    return STATUS_OK


def tree_verify_attn(q_bits, k_bits, v_bits, page_table, prefix_len, n_nodes, parents,
                     scale, page_size=16, rows=None):
    """Tree-masked attention of every tree node over its request's paged cache.

    For request b, query head h and node i, the visible keys are the prefix
    positions 0..L-1 and the tree positions L+j for every j that is an
    ancestor of i or i itself (the mask M of Tech Radar section 2).  The tree's
    own K/V already sit at positions L..L+N-1 of the request's pages.  Query
    head h reads KV head h // G with G = Hq / Hkv.

        s_t = scale * <q, k_t>,   o = sum_t softmax(s)_t v_t,
        lse = log sum_t exp(s_t)  (natural log).

    Inputs are raw bf16 bits (uint16): q [B, n_max, Hq, D],
    caches [num_pages, Hkv, page_size, D]; page_table int32 [B, max_pages].
    ``rows`` optionally restricts the work to a list of (b, i, h) triples.

    Returns (out float64 [B, n_max, Hq, D], lse float64 [B, n_max, Hq],
    status int32 [B]); entries not computed are NaN.
    """
    B, n_max, Hq, D = q_bits.shape
    num_pages, Hkv = k_bits.shape[0], k_bits.shape[1]
    G = Hq // Hkv
    out = np.full((B, n_max, Hq, D), np.nan)
    lse = np.full((B, n_max, Hq), np.nan)
    status = np.zeros(B, dtype=np.int32)

    if rows is None:
        wanted = {b: None for b in range(B)}
    else:
        wanted = {}
        for (b, i, h) in rows:
            wanted.setdefault(int(b), []).append((int(i), int(h)))

    for b, sel in wanted.items():
        L, N = int(prefix_len[b]), int(n_nodes[b])
        st = _request_pages_ok(page_table[b], L, N, num_pages, page_size)
        if not tree_is_valid(parents[b], N):
            st |= STATUS_BAD_TREE
        status[b] = st
        if st != STATUS_OK:
            continue
        pairs = sel if sel is not None else [(i, h) for i in range(N) for h in range(Hq)]
        by_node = {}
        for (i, h) in pairs:
            by_node.setdefault(i, []).append(h)
        for i, heads in by_node.items():
            # the explicit key sequence of node i: prefix, then its root-to-node path
            positions = list(range(L)) + [L + j for j in ancestors_or_self(parents[b], i)]
            pos = np.asarray(positions, dtype=np.int64)
            page = np.asarray(page_table[b])[pos // page_size]
            slot = pos % page_size
            K = bf16_to_f64(k_bits[page, :, slot, :])   # [T, Hkv, D]
            Vv = bf16_to_f64(v_bits[page, :, slot, :])  # [T, Hkv, D]
            for h in heads:
                g = h // G
                qv = bf16_to_f64(q_bits[b, i, h])       # [D]
                s = scale * (K[:, g, :] @ qv)           # [T]
                m = np.max(s)
                w = np.exp(s - m)
                out[b, i, h] = (w @ Vv[:, g, :]) / np.sum(w)
                lse[b, i, h] = m + np.log(np.sum(w))
    return out, lse, status


# --------------------------------------------------------------------------
# step 3a: greedy acceptance
# --------------------------------------------------------------------------
def _first_argmax(row) -> int:
    """Largest entry, lowest index on ties (numpy.argmax semantics)."""
    return int(np.argmax(np.asarray(row)))


def tree_accept_greedy(target_logits, tokens, parents, n_nodes, V=None):
    """Greedy (T = 0) acceptance of the longest matching root-to-node path.

    A non-root node j "hits" when its token equals the target's argmax at its
    parent (the drafter's argmax rule of Tech Radar section 2 applied to the
    target).  A node c is accepted when every non-root node on its
    root-to-node path hits.  The result is the accepted node of largest depth
    (lowest index on ties); the emitted tokens are the path's drafted tokens
    followed by the target's argmax at the result node (k hits emit k+1
    tokens: study note, case 1).

    Returns dict with accept_len int32 [B], path_nodes int32 [B, n_max]
    (root first, -1 padded), out_tokens int32 [B, n_max+1] (-1 padded),
    status int32 [B].
    """
    B, n_max, Vdim = target_logits.shape
    V = Vdim if V is None else V
    accept_len = np.zeros(B, dtype=np.int32)
    path_nodes = np.full((B, n_max), -1, dtype=np.int32)
    out_tokens = np.full((B, n_max + 1), -1, dtype=np.int32)
    status = np.zeros(B, dtype=np.int32)
    for b in range(B):
        n = int(n_nodes[b])
        if not tree_is_valid(parents[b], n):
            status[b] = STATUS_BAD_TREE
            continue
        if any(not (0 <= int(tokens[b, c]) < V) for c in range(1, n)):
            status[b] = STATUS_BAD_TOKEN
            continue
        best, best_depth = 0, 0
        for c in range(n):
            path = ancestors_or_self(parents[b], c)
            ok = all(int(tokens[b, j]) == _first_argmax(target_logits[b, int(parents[b, j])])
                     for j in path[1:])
            if ok and len(path) - 1 > best_depth:
                best, best_depth = c, len(path) - 1
        path = ancestors_or_self(parents[b], best)
        accept_len[b] = best_depth
        path_nodes[b, : len(path)] = path
        emitted = [int(tokens[b, j]) for j in path[1:]] + [_first_argmax(target_logits[b, best])]
        out_tokens[b, : len(emitted)] = emitted
    return dict(accept_len=accept_len, path_nodes=path_nodes, out_tokens=out_tokens,
                status=status)


# --------------------------------------------------------------------------
# step 3b: rejection-sampling acceptance
# --------------------------------------------------------------------------
def softmax_t(z, T):
    """softmax(z / T) in fp64."""
    x = np.asarray(z, dtype=np.float64) / T
    e = np.exp(x - np.max(x))
    return e / np.sum(e)


def node_plan(p, q, child_tokens):
    """The acceptance plan at one tree node (multi-child reading of the
    rejection rule): children are tried in the given (ascending node) order;
    child k with token x is accepted with probability min(1, cur_k(x)/q(x))
    where cur_0 = p and, after a rejection, cur_{k+1} = max(0, cur_k - q)
    normalised (left unchanged if that residual sums to zero).

    Returns (cur_list, final) where cur_list[k] is the distribution the k-th
    child is tested against and ``final`` the one the bonus token is drawn
    from when every child is rejected.
    """
    cur = np.asarray(p, dtype=np.float64)
    q = np.asarray(q, dtype=np.float64)
    cur_list = []
    for _x in child_tokens:
        cur_list.append(cur)
        r = np.maximum(0.0, cur - q)
        s = np.sum(r)
        cur = r / s if s > 0 else cur
    return cur_list, cur


def node_plan_wor(p, q, child_tokens):
    """The acceptance plan at one tree node for siblings drafted without
    replacement (top-k style trees whose siblings are distinct tokens): as
    ``node_plan``, but after child k with token x is rejected the draft is
    also updated, q_{k+1} = q_k with x removed and renormalised (all zero if
    nothing is left).  The target side is unchanged: cur_{k+1} = max(0,
    cur_k - q_k) normalised, with q_k the draft child k was tested against.

    Sequential rejection with q renormalised after each removal is the
    standard recursive rejection sampling for draws without replacement: the
    k-th sibling is a draw from q_k, so each step is an ordinary
    speculative-sampling step against the current residual.

    Returns (plans, final): plans[k] = (cur_k, q_k) for the k-th child and
    ``final`` the distribution the bonus token is drawn from when every child
    is rejected.
    """
    cur = np.asarray(p, dtype=np.float64)
    qk = np.asarray(q, dtype=np.float64)
    plans = []
    for x in child_tokens:
        plans.append((cur, qk))
        r = np.maximum(0.0, cur - qk)
        s = np.sum(r)
        cur = r / s if s > 0 else cur
        q_next = qk.copy()
        q_next[int(x)] = 0.0
        sq = np.sum(q_next)
        qk = q_next / sq if sq > 0 else q_next
    return plans, cur


def accept_test(u, cur_x, q_x):
    """Accept iff u * q(x) < cur(x), i.e. u < min(1, cur(x)/q(x)) without a
    division; with q(x) = 0 this accepts iff cur(x) > 0."""
    return u * q_x < cur_x


def inverse_cdf(w, u):
    """First index j with u * S < C_j, C_j = sum_{v<=j} w_v, S = C_{V-1}
    (zero-weight entries are never chosen).  Returns (j, margin) where margin
    is min |u*S - C| over C_{j-1}, C_j relative to S."""
    C = np.cumsum(np.asarray(w, dtype=np.float64))
    S = C[-1]
    t = u * S
    j = int(np.searchsorted(C, t, side="right"))
    if j >= len(C):                       # u*S >= S only through rounding
        j = int(np.nonzero(np.asarray(w) > 0)[0][-1])
    lo = C[j - 1] if j > 0 else 0.0
    margin = min(abs(t - C[j]), abs(t - lo)) / S
    return j, margin


def tree_accept_sampling(target_logits, draft_logits, tokens, parents, n_nodes, temperature,
                         u_accept, u_sample, V=None, without_replacement=False):
    """Rejection-sampling acceptance at temperature T > 0 (lossless
    verification: troisinh.com "Why it works"; study note case 3).

    Walk from the root.  At node n set p = softmax(target[n]/T),
    q = softmax(draft[n]/T) (draft row n is the distribution n's children were
    drawn from).  Children c of n are tried in ascending index with
    u = u_accept[c]; the first accepted child becomes the next node.  If no
    child is accepted (or n is a leaf) the bonus token is drawn from the
    current distribution (the residual after the rejections, or p at a leaf)
    by inverse CDF with u = u_sample[n], and the walk ends.

    ``without_replacement`` selects the sibling rule of ``node_plan_wor`` (the
    draft renormalised without each rejected sibling's token) instead of
    ``node_plan`` (draft fixed).

    Returns dict like ``tree_accept_greedy`` plus ``near_boundary`` bool [B]:
    some decision of the walk had |u - cur(x)/q(x)| < 1e-6 or an inverse-CDF
    margin below 1e-6, where a rounding difference may legitimately change the
    outcome.
    """
    B, n_max, Vdim = target_logits.shape
    V = Vdim if V is None else V
    T = float(temperature)
    accept_len = np.zeros(B, dtype=np.int32)
    path_nodes = np.full((B, n_max), -1, dtype=np.int32)
    out_tokens = np.full((B, n_max + 1), -1, dtype=np.int32)
    status = np.zeros(B, dtype=np.int32)
    near = np.zeros(B, dtype=bool)
    for b in range(B):
        n_b = int(n_nodes[b])
        if not tree_is_valid(parents[b], n_b):
            status[b] = STATUS_BAD_TREE
            continue
        if any(not (0 <= int(tokens[b, c]) < V) for c in range(1, n_b)):
            status[b] = STATUS_BAD_TOKEN
            continue
        kids = [[] for _ in range(n_b)]
        for c in range(1, n_b):
            kids[int(parents[b, c])].append(c)
        node, path, emitted = 0, [0], []
        while True:
            p = softmax_t(target_logits[b, node], T)
            q = softmax_t(draft_logits[b, node], T)
            child_tokens = [int(tokens[b, c]) for c in kids[node]]
            if without_replacement:
                plans, final = node_plan_wor(p, q, child_tokens)
            else:
                cur_list, final = node_plan(p, q, child_tokens)
                plans = [(cur, q) for cur in cur_list]
            nxt = None
            for c, x, (cur, qk) in zip(kids[node], child_tokens, plans):
                u = float(u_accept[b, c])
                if qk[x] > 0 and abs(u - cur[x] / qk[x]) < NEAR_BOUNDARY:
                    near[b] = True
                if accept_test(u, cur[x], qk[x]):
                    nxt = c
                    break
            if nxt is not None:
                node = nxt
                path.append(node)
                emitted.append(int(tokens[b, node]))
                continue
            j, margin = inverse_cdf(final, float(u_sample[b, node]))
            if margin < NEAR_BOUNDARY:
                near[b] = True
            emitted.append(j)
            break
        accept_len[b] = len(path) - 1
        path_nodes[b, : len(path)] = path
        out_tokens[b, : len(emitted)] = emitted
    return dict(accept_len=accept_len, path_nodes=path_nodes, out_tokens=out_tokens,
                status=status, near_boundary=near)


# --------------------------------------------------------------------------
# step 4: KV commit of the accepted path
# --------------------------------------------------------------------------
def kv_commit_path(k_layers, v_layers, page_table, prefix_len, n_nodes, accept_len, path_nodes,
                   page_size=16):
    """Keep the accepted branch's K/V and drop the rest (Tech Radar section 2,
    sequence diagram): for k = 1..a, the K and V rows of logical position
    L + path[k] move to position L + k in every layer and KV head; the root
    stays at L.  The new length is L + a + 1 and the committed physical slots
    are page_table[(L+k)//P]*P + (L+k)%P for k = 0..a.

    Caches are given per layer as [n_layers, num_pages, Hkv, P, D] arrays of
    any dtype; copies are returned.  Moves are applied in increasing k, which
    reads every source before it can be overwritten (path[k] >= k).

    Returns (k_new, v_new, committed_slots int64 [B, n_max] (-1 padded),
    new_len int32 [B], status int32 [B]).
    """
    k_new = np.array(k_layers, copy=True)
    v_new = np.array(v_layers, copy=True)
    B, n_max = path_nodes.shape
    num_pages = k_new.shape[1]
    slots = np.full((B, n_max), -1, dtype=np.int64)
    new_len = np.zeros(B, dtype=np.int32)
    status = np.zeros(B, dtype=np.int32)
    for b in range(B):
        L, N, a = int(prefix_len[b]), int(n_nodes[b]), int(accept_len[b])
        st = _request_pages_ok(page_table[b], L, N, num_pages, page_size)
        path = [int(x) for x in path_nodes[b, : max(a, 0) + 1]]
        if N < 1 or N > n_max or a < 0 or a >= N or path[0] != 0 or \
                any(path[k] >= N for k in range(a + 1)) or \
                any(path[k] <= path[k - 1] for k in range(1, a + 1)):
            st |= STATUS_BAD_TREE
        status[b] = st
        if st != STATUS_OK:
            new_len[b] = L
            continue
        for k in range(1, a + 1):
            src, dst = L + path[k], L + k
            if src == dst:
                continue
            sp, so = int(page_table[b, src // page_size]), src % page_size
            dp, do = int(page_table[b, dst // page_size]), dst % page_size
            k_new[:, dp, :, do, :] = k_new[:, sp, :, so, :]
            v_new[:, dp, :, do, :] = v_new[:, sp, :, so, :]
        for k in range(a + 1):
            pos = L + k
            slots[b, k] = int(page_table[b, pos // page_size]) * page_size + pos % page_size
        new_len[b] = L + a + 1
    return k_new, v_new, slots, new_len, status


# --------------------------------------------------------------------------
# step 0: dynamic tree expansion (the drafting loop before verification)
# --------------------------------------------------------------------------
NEAR_EXPAND = 1e-4


def draft_entropy(z):
    """H = -sum_i P(x_i) log P(x_i) with P = softmax(z), natural log (Tech
    Radar section 2, "Dynamic Tree-Attention Masking", the entropy of the
    draft distribution).  Terms with P = 0 contribute 0."""
    x = np.asarray(z, dtype=np.float64)
    x = x - np.max(x)
    log_p = x - np.log(np.sum(np.exp(x)))
    p = np.exp(log_p)
    return float(-np.sum(np.where(p > 0.0, p * log_p, 0.0)))


def branch_width(H, top_k):
    """Children a frontier node gets: round(e^H) clamped to [1, top_k].

    Reading of the same passage: low entropy extends a single branch, high
    entropy widens the tree up to 8 nodes.  e^H is the perplexity, the number
    of equally likely tokens with the same entropy, so the plainest continuous
    rule is its nearest integer.  The step from w to w + 1 children sits at
    H = ln(w + 1/2); the width is 1 plus the number of those thresholds
    (w = 1 .. top_k - 1) that H reaches.
    """
    w = 1
    for j in range(1, top_k):
        if H >= np.log(j + 0.5):
            w = j + 1
    return w


def top_tokens(z, w):
    """The w most probable tokens of a draft row, most probable first; equal
    logits in ascending token id (top-k expansion of the drafter): w rounds
    of taking the first maximum among the tokens not yet taken."""
    z = np.array(z, dtype=np.float64, copy=True)
    picked = []
    for _ in range(min(w, len(z))):
        t = int(np.argmax(z))                 # first index of the maximum
        picked.append(t)
        z[t] = -np.inf
    return picked


def log_softmax_at(z, t):
    """log P(t) for P = softmax(z), in fp64."""
    x = np.asarray(z, dtype=np.float64)
    m = np.max(x)
    return float(x[t] - m - np.log(np.sum(np.exp(x - m))))


def tree_expand_level(draft_logits, parents, tokens, scores, n_nodes, level_start, top_k, max_new,
                      budget):
    """One level of the dynamic expansion loop (Tech Radar section 2, sequence
    diagram: per depth, the drafter scores entropy, then beam search prunes
    the low branches; the tree holds at most 64 nodes).

    State per request b: nodes [0, n_nodes[b]) with parents, tokens and
    cumulative log-probabilities ``scores``; the frontier is the last level
    added, nodes [level_start[b], n_nodes[b]).  Draft row f of
    ``draft_logits[b]`` is the drafter's distribution over the children of
    node f (the same row later serves as the q row of verification).

    For each frontier node f (ascending): P = softmax(draft row f),
    H_f = draft_entropy, w_f = branch_width(H_f, top_k); its top w_f tokens
    are candidates (f, r, token, score_f + log P(token)).  Beam step: of all
    candidates the best  keep = min(max_new, budget - n_nodes, count)  by
    score are kept (equal scores: lower f, then lower rank r) and appended as
    nodes n_nodes, n_nodes + 1, ... in (f, r) order, so parents precede
    children and siblings are contiguous, most probable first.  Afterwards
    level_start = old n_nodes and n_nodes grows by ``keep``.

    An invalid state (not 1 <= n_nodes <= n_max, or not 0 <= level_start <=
    n_nodes) leaves the request unchanged with STATUS_BAD_TREE.

    Returns dict(parents, tokens, scores, n_nodes, level_start: the new state
    (copies), entropy / width: per frontier node (NaN / 0 elsewhere), status,
    near_boundary: some entropy lies within NEAR_EXPAND of a width threshold
    or the last kept and first dropped scores are within NEAR_EXPAND, where a
    rounding difference may legitimately change the result).
    """
    parents = np.array(parents, dtype=np.int32, copy=True)
    tokens = np.array(tokens, dtype=np.int32, copy=True)
    scores = np.array(scores, dtype=np.float64, copy=True)
    n_nodes = np.array(n_nodes, dtype=np.int32, copy=True)
    level_start = np.array(level_start, dtype=np.int32, copy=True)
    B, n_max = parents.shape
    entropy = np.full((B, n_max), np.nan)
    width = np.zeros((B, n_max), dtype=np.int32)
    status = np.zeros(B, dtype=np.int32)
    near = np.zeros(B, dtype=bool)
    for b in range(B):
        n, ls = int(n_nodes[b]), int(level_start[b])
        if not (1 <= n <= n_max and 0 <= ls <= n):
            status[b] = STATUS_BAD_TREE
            continue
        cands = []                                   # (score, f, r, token)
        for f in range(ls, n):
            row = draft_logits[b, f]
            H = draft_entropy(row)
            w = branch_width(H, top_k)
            entropy[b, f], width[b, f] = H, w
            for j in range(1, top_k):
                if abs(H - np.log(j + 0.5)) < NEAR_EXPAND:
                    near[b] = True
            for r, t in enumerate(top_tokens(row, w)):
                cands.append((float(scores[b, f]) + log_softmax_at(row, t), f, r, t))
        keep = max(0, min(max_new, budget - n, len(cands)))
        # beam: repeatedly take the best remaining candidate
        remaining = list(cands)
        chosen = []
        for _ in range(keep):
            best = 0
            for k in range(1, len(remaining)):
                s, f, r, _t = remaining[k]
                sb, fb, rb, _tb = remaining[best]
                if s > sb or (s == sb and (f, r) < (fb, rb)):
                    best = k
            chosen.append(remaining.pop(best))
        if chosen and remaining:
            first_out = max(c[0] for c in remaining)
            if abs(chosen[-1][0] - first_out) < NEAR_EXPAND * max(1.0, abs(first_out)):
                near[b] = True
        chosen.sort(key=lambda c: (c[1], c[2]))
        for k, (s, f, _r, t) in enumerate(chosen):
            parents[b, n + k] = f
            tokens[b, n + k] = t
            scores[b, n + k] = s
        level_start[b] = n
        n_nodes[b] = n + keep
    return dict(parents=parents, tokens=tokens, scores=scores, n_nodes=n_nodes,
                level_start=level_start, entropy=entropy, width=width, status=status,
                near_boundary=near)


def tree_build_dynamic(draft_logits, root_tokens, n_levels, top_k, max_new, budget):
    """The whole expansion loop: a root per request (token root_tokens[b],
    score 0), then ``n_levels`` calls of tree_expand_level (depth 4-6 in the
    pages).  draft_logits [B, n_max, V] holds the drafter's row for every node
    id that may be created.  Returns the final state of tree_expand_level
    with near_boundary OR-ed over the levels and entropy / width of every
    expanded node."""
    B, n_max, _V = draft_logits.shape
    parents = np.full((B, n_max), -1, dtype=np.int32)
    tokens = np.zeros((B, n_max), dtype=np.int32)
    tokens[:, 0] = np.asarray(root_tokens, dtype=np.int32)
    scores = np.zeros((B, n_max), dtype=np.float64)
    n_nodes = np.ones(B, dtype=np.int32)
    level_start = np.zeros(B, dtype=np.int32)
    entropy = np.full((B, n_max), np.nan)
    width = np.zeros((B, n_max), dtype=np.int32)
    near = np.zeros(B, dtype=bool)
    status = np.zeros(B, dtype=np.int32)
    for _ in range(n_levels):
        out = tree_expand_level(draft_logits, parents, tokens, scores, n_nodes, level_start, top_k,
                                max_new, budget)
        parents, tokens, scores = out["parents"], out["tokens"], out["scores"]
        n_nodes, level_start = out["n_nodes"], out["level_start"]
        got = ~np.isnan(out["entropy"])
        entropy[got] = out["entropy"][got]
        width[got] = out["width"][got]
        near |= out["near_boundary"]
        status |= out["status"]
    return dict(parents=parents, tokens=tokens, scores=scores, n_nodes=n_nodes,
                level_start=level_start, entropy=entropy, width=width, status=status,
                near_boundary=near)


# --------------------------------------------------------------------------
# step 5: zero-copy pruning of the rejected branches' pages
# --------------------------------------------------------------------------
def kv_prune_pages(page_table, refcount, prefix_len, n_nodes, new_len, status_in=None, page_size=16):
    """Release, without copying anything, the pages that after the commit
    hold only rejected tree rows (Tech Radar, failure mode 2: rejected
    branches leave garbage blocks in the page table; managing the branches as
    a prefix tree frees them at once, with no copy).

    After the commit request b keeps positions [0, new_len); positions
    [new_len, L + N) held the tree and are garbage.  Page-table slots
    s = ceil(new_len / P) .. ceil((L + N) / P) - 1 contain no kept position,
    so the request lets go of them: the slot becomes -1 and the physical
    page's reference count drops by one; a page whose count reaches zero is
    free (pages shared with other sequences, counts above one, stay in use).
    The slot holding position new_len - 1 and everything before it are kept.

    Requests are handled in index order; the final counts and the set of
    freed pages do not depend on that order for valid inputs.  A request is
    skipped when its incoming status is non-zero; BAD_TREE when new_len is
    not in [L + 1, L + N]; CAPACITY when L + N does not fit the row (or
    L < 0); PAGE_OOB when a released slot's id is outside [0, num_pages)
    (nothing released); BAD_REFCOUNT when a released page's count is already
    zero (that slot is cleared, the count stays zero).

    Returns (page_table copy, refcount copy, freed: sorted list of page ids,
    status int32 [B]).
    """
    pt = np.array(page_table, dtype=np.int32, copy=True)
    rc = np.array(refcount, dtype=np.int32, copy=True)
    B, max_pages = pt.shape
    num_pages = rc.shape[0]
    status = np.zeros(B, dtype=np.int32)
    freed = []
    for b in range(B):
        if status_in is not None and int(status_in[b]) != 0:
            status[b] = int(status_in[b])
            continue
        L, N, nl = int(prefix_len[b]), int(n_nodes[b]), int(new_len[b])
        if L < 0 or N < 1 or (L + N + page_size - 1) // page_size > max_pages:
            status[b] = STATUS_CAPACITY
            continue
        if not (L + 1 <= nl <= L + N):
            status[b] = STATUS_BAD_TREE
            continue
        first = (nl + page_size - 1) // page_size
        last = (L + N + page_size - 1) // page_size
        slots = list(range(first, last))
        if any(not (0 <= int(pt[b, s]) < num_pages) for s in slots):
            status[b] = STATUS_PAGE_OOB
            continue
        for s in slots:
            pid = int(pt[b, s])
            pt[b, s] = -1
            if rc[pid] <= 0:
                status[b] |= STATUS_BAD_REFCOUNT
                continue
            rc[pid] -= 1
            if rc[pid] == 0:
                freed.append(pid)
    return pt, rc, sorted(freed), status


# --------------------------------------------------------------------------
# low-bit KV: verify attention over a 4-bit cache
# --------------------------------------------------------------------------
Q4_GROUP = 32


def f64_to_bf16_bits_via_f32(x):
    """Round to float32 (nearest even), then to bfloat16 (nearest even);
    returns the bf16 bit patterns (uint16)."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def dequantize_q4(codes, params):
    """Decode a 4-bit KV cache to bf16 rows (troisinh.com "EAGLE - Draft head
    ...": EAGLE pairs with an INT4 KV cache, and its further-reading list
    names KV-cache quantisation to INT4/INT3).

    codes  uint8 [..., D/2]: byte j holds dims 2j (low nibble) and 2j+1 (high
           nibble), unsigned codes 0..15;
    params float16 [..., 2 * D / 32]: (scale, zero) of each group of 32 dims.
    Value of dim d: bf16(fp32(code * scale + zero)) for the group of d (the
    product and sum exact in fp64, one rounding to fp32, one to bf16).
    Returns bf16 bit patterns uint16 [..., D].
    """
    codes = np.asarray(codes, dtype=np.uint8)
    D = codes.shape[-1] * 2
    c = np.empty(codes.shape[:-1] + (D,), dtype=np.float64)
    c[..., 0::2] = (codes & 0x0F).astype(np.float64)
    c[..., 1::2] = (codes >> 4).astype(np.float64)
    prm = np.asarray(params, dtype=np.float16).astype(np.float64)
    n_groups = D // Q4_GROUP
    scale = np.repeat(prm[..., 0:2 * n_groups:2], Q4_GROUP, axis=-1)
    zero = np.repeat(prm[..., 1:2 * n_groups:2], Q4_GROUP, axis=-1)
    return f64_to_bf16_bits_via_f32(c * scale + zero)


def tree_verify_attn_q4(q_bits, k_codes, k_params, v_codes, v_params, page_table, prefix_len, n_nodes,
                        parents, scale, page_size=16, rows=None):
    """Tree-masked attention over a 4-bit paged cache: the cache decoded by
    ``dequantize_q4`` (caches [num_pages, Hkv, page_size, D/2] codes and
    [num_pages, Hkv, page_size, 2 * D / 32] params), then ``tree_verify_attn``."""
    return tree_verify_attn(q_bits, dequantize_q4(k_codes, k_params), dequantize_q4(v_codes, v_params),
                            page_table, prefix_len, n_nodes, parents, scale, page_size=page_size, rows=rows)


def quantize_q4(x_bits):
    """Encode bf16 rows (uint16 bits [..., D]) in the 4-bit format that
    ``dequantize_q4`` decodes.  Per row and group of 32 dims, in fp32 IEEE
    arithmetic (round to nearest even at each step) with fp16 parameters:
        zero  = fp16(min x)
        scale = fp16((max x - min x) / 15)
        inv   = fp32(1 / scale)
        code  = clamp(rint((x - zero) * inv), 0, 15)   (0 when scale is 0)
    Codes are integer decisions taken from floating point, so the arithmetic
    and its rounding order are part of the definition.  Returns (codes uint8
    [..., D/2], params float16 [..., 2 * D / 32])."""
    x = bf16_to_f64(x_bits).astype(np.float32)
    D = x.shape[-1]
    g = D // Q4_GROUP
    xg = x.reshape(x.shape[:-1] + (g, Q4_GROUP))
    mn = xg.min(axis=-1)
    mx = xg.max(axis=-1)
    zero = mn.astype(np.float16)
    scale = ((mx - mn) / np.float32(15.0)).astype(np.float16)
    z32 = zero.astype(np.float32)[..., None]
    s32 = scale.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.float32(1.0) / s32
        q = np.rint((xg - z32) * inv)
    q = np.where(s32 > 0, q, 0.0)
    q = np.clip(q, 0, 15).astype(np.uint8).reshape(x.shape)
    codes = (q[..., 0::2] | (q[..., 1::2] << 4)).astype(np.uint8)
    params = np.empty(x.shape[:-1] + (2 * g,), dtype=np.float16)
    params[..., 0::2] = scale
    params[..., 1::2] = zero
    return codes, params


# --------------------------------------------------------------------------
# low-bit KV: verify attention over a 3-bit cache
# --------------------------------------------------------------------------
def q3_code_values(codes, D):
    """The integer codes 0..7 of a 3-bit row layout (uint8 [..., 3 * D / 8]),
    as int64 [..., D].  Bytes [0, D/4) hold the low two bits of every code,
    four per byte: byte j holds dims 4j .. 4j+3, dim 4j+i in bits 2i, 2i+1.
    Bytes [D/4, 3D/8) hold the third bit of every code, eight per byte: byte
    D/4 + j holds dims 8j .. 8j+7, dim 8j+i in bit i."""
    codes = np.asarray(codes, dtype=np.uint8)
    lo = codes[..., : D // 4].astype(np.int64)
    hi = codes[..., D // 4: 3 * D // 8].astype(np.int64)
    c = np.empty(codes.shape[:-1] + (D,), dtype=np.int64)
    for i in range(4):
        c[..., i::4] = (lo >> (2 * i)) & 3
    for i in range(8):
        c[..., i::8] |= ((hi >> i) & 1) << 2
    return c


def q3_pack(c):
    """Inverse of ``q3_code_values``: int codes 0..7 [..., D] -> uint8 [..., 3D/8]."""
    c = np.asarray(c, dtype=np.int64)
    D = c.shape[-1]
    out = np.zeros(c.shape[:-1] + (3 * D // 8,), dtype=np.int64)
    for i in range(4):
        out[..., : D // 4] |= (c[..., i::4] & 3) << (2 * i)
    for i in range(8):
        out[..., D // 4:] |= ((c[..., i::8] >> 2) & 1) << i
    return out.astype(np.uint8)


def dequantize_q3(codes, params):
    """Decode a 3-bit KV cache to bf16 rows (troisinh.com "EAGLE - Draft head
    ...": its further-reading list names KV-cache quantisation to INT4/INT3).

    codes  uint8 [..., 3 * D / 8] in the layout of ``q3_code_values``, codes 0..7;
    params float16 [..., 2 * D / 32]: (scale, zero) of each group of 32 dims.
    Value of dim d: bf16(fp32(code * scale + zero)) for the group of d (the
    product and sum exact in fp64, one rounding to fp32, one to bf16), as for
    the 4-bit format.  Returns bf16 bit patterns uint16 [..., D].
    """
    codes = np.asarray(codes, dtype=np.uint8)
    D = codes.shape[-1] * 8 // 3
    c = q3_code_values(codes, D).astype(np.float64)
    prm = np.asarray(params, dtype=np.float16).astype(np.float64)
    n_groups = D // Q4_GROUP
    scale = np.repeat(prm[..., 0:2 * n_groups:2], Q4_GROUP, axis=-1)
    zero = np.repeat(prm[..., 1:2 * n_groups:2], Q4_GROUP, axis=-1)
    return f64_to_bf16_bits_via_f32(c * scale + zero)


def tree_verify_attn_q3(q_bits, k_codes, k_params, v_codes, v_params, page_table, prefix_len, n_nodes,
                        parents, scale, page_size=16, rows=None):
    """Tree-masked attention over a 3-bit paged cache: the cache decoded by
    ``dequantize_q3`` (caches [num_pages, Hkv, page_size, 3 * D / 8] codes and
    [num_pages, Hkv, page_size, 2 * D / 32] params), then ``tree_verify_attn``."""
    return tree_verify_attn(q_bits, dequantize_q3(k_codes, k_params), dequantize_q3(v_codes, v_params),
                            page_table, prefix_len, n_nodes, parents, scale, page_size=page_size, rows=rows)


def quantize_q3(x_bits):
    """Encode bf16 rows (uint16 bits [..., D]) in the 3-bit format that
    ``dequantize_q3`` decodes.  Per row and group of 32 dims, in fp32 IEEE
    arithmetic (round to nearest even at each step) with fp16 parameters, as
    the 4-bit encoder with 8 levels:
        zero  = fp16(min x)
        scale = fp16((max x - min x) / 7)
        inv   = fp32(1 / scale)
        code  = clamp(rint((x - zero) * inv), 0, 7)   (0 when scale is 0)
    Returns (codes uint8 [..., 3 * D / 8], params float16 [..., 2 * D / 32])."""
    x = bf16_to_f64(x_bits).astype(np.float32)
    D = x.shape[-1]
    g = D // Q4_GROUP
    xg = x.reshape(x.shape[:-1] + (g, Q4_GROUP))
    mn = xg.min(axis=-1)
    mx = xg.max(axis=-1)
    zero = mn.astype(np.float16)
    scale = ((mx - mn) / np.float32(7.0)).astype(np.float16)
    z32 = zero.astype(np.float32)[..., None]
    s32 = scale.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.float32(1.0) / s32
        q = np.rint((xg - z32) * inv)
    q = np.where(s32 > 0, q, 0.0)
    q = np.clip(q, 0, 7).astype(np.int64).reshape(x.shape)
    params = np.empty(x.shape[:-1] + (2 * g,), dtype=np.float16)
    params[..., 0::2] = scale
    params[..., 1::2] = zero
    return q3_pack(q), params
