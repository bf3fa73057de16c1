"""GPU parity of tv_tree_expand (one level of dynamic tree construction)
against the oracle.

Each level runs on the GPU from the GPU's own state; the oracle runs the same
level from that same state (fp32 scores widened to fp64).  The new nodes
(parents, tokens), n_nodes, level_start and the widths must be bit-exact and
the scores and entropies within fp32 accumulation error, except in requests
where the oracle reports a decision within 1e-4 of its threshold (an entropy
at a width step, or equal-looking scores at the beam cut): those are counted
and must stay rare.
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
from eagle_speculative_decoding_attn_gb300 import workloads as W
from golden_io import read_fixture
from gpu_helpers import require_gpu, to_dev

pytestmark = pytest.mark.gpu

SCORE_ATOL, SCORE_RTOL = 1e-4, 1e-5   # cumulative log-probabilities (fp32, <= 6 terms)
ENTROPY_ATOL = 2e-4                   # fp32 sums of up to 128256 terms


class DevTree:
    """The expansion state of B requests on the device, started at a root."""

    def __init__(self, logits, root_tokens, dev, n_max):
        B = logits.shape[0]
        self.logits = to_dev(logits, dev)
        self.parents = torch.full((B, n_max), -1, dtype=torch.int32, device=dev)
        self.tokens = torch.zeros((B, n_max), dtype=torch.int32, device=dev)
        self.tokens[:, 0] = to_dev(np.asarray(root_tokens, dtype=np.int32), dev)
        self.scores = torch.zeros((B, n_max), dtype=torch.float32, device=dev)
        self.n_nodes = torch.ones(B, dtype=torch.int32, device=dev)
        self.level_start = torch.zeros(B, dtype=torch.int32, device=dev)
        self.status = torch.zeros(B, dtype=torch.int32, device=dev)
        self.entropy = torch.full((B, n_max), float("nan"), dtype=torch.float32, device=dev)
        self.width = torch.zeros((B, n_max), dtype=torch.int32, device=dev)

    def state(self):
        return {k: getattr(self, k).cpu().numpy().copy() for k in
                ("parents", "tokens", "scores", "n_nodes", "level_start", "status", "entropy", "width")}

    def level(self, top_k, max_new, budget, max_frontier=None, workspace=None):
        tvb.tree_expand(self.logits, self.parents, self.tokens, self.scores, self.n_nodes, self.level_start,
                        self.status, top_k=top_k, max_new=max_new, budget=budget, max_frontier=max_frontier,
                        entropy=self.entropy, width=self.width, workspace=workspace)
        torch.cuda.synchronize()


def _compare_level(before, after, logits, top_k, max_new, budget):
    """Oracle level from the GPU's input state; returns the near-boundary flags."""
    ref = oracle.tree_expand_level(logits, before["parents"], before["tokens"], before["scores"].astype(np.float64),
                                   before["n_nodes"], before["level_start"], top_k, max_new, budget)
    near = ref["near_boundary"]
    assert np.array_equal(after["status"], ref["status"])
    for b in range(logits.shape[0]):
        ls, n0 = int(before["level_start"][b]), int(before["n_nodes"][b])
        fr = slice(ls, n0)
        if ref["status"][b] == 0 and n0 < budget:
            np.testing.assert_allclose(after["entropy"][b, fr], ref["entropy"][b, fr], rtol=0, atol=ENTROPY_ATOL)
        if near[b]:
            continue
        assert after["n_nodes"][b] == ref["n_nodes"][b], b
        assert after["level_start"][b] == ref["level_start"][b], b
        n1 = int(ref["n_nodes"][b])
        assert after["parents"][b, :n1].tolist() == ref["parents"][b, :n1].tolist(), b
        assert after["tokens"][b, :n1].tolist() == ref["tokens"][b, :n1].tolist(), b
        np.testing.assert_allclose(after["scores"][b, n0:n1], ref["scores"][b, n0:n1], rtol=SCORE_RTOL,
                                   atol=SCORE_ATOL)
        if ref["status"][b] == 0 and n0 < budget:
            assert after["width"][b, fr].tolist() == ref["width"][b, fr].tolist(), b
    return near


def _grow_and_compare(wl, dev, n_levels=None, max_frontier=None):
    tree = DevTree(wl.draft_logits, wl.root_tokens, dev, wl.n_max)
    near_count, rows = 0, 0
    for _ in range(wl.n_levels if n_levels is None else n_levels):
        before = tree.state()
        tree.level(wl.top_k, wl.max_new, wl.budget, max_frontier=max_frontier)
        after = tree.state()
        near = _compare_level(before, after, wl.draft_logits, wl.top_k, wl.max_new, wl.budget)
        near_count += int(near.sum())
        rows += int(np.sum(before["n_nodes"] - before["level_start"]))
    return tree.state(), near_count, rows


def test_hand_worked_example():
    dev = require_gpu()
    fx = read_fixture("expand_example.txt")
    V, top_k = int(fx["V"][0]), int(fx["top_k"][0])
    rows = np.zeros((2, 8, V), dtype=np.float32)
    for f in range(4):
        rows[:, f] = [float(x) for x in fx[f"row{f}"]]
    ints = lambda key: [int(x) for x in fx[key]]
    floats = lambda key: [float(x) for x in fx[key]]
    for case, budget in (("caseA", 8), ("caseB", 6)):
        tree = DevTree(rows, [0, 0], dev, 8)
        tree.level(top_k, 3, budget)
        tree.level(top_k, 4, budget, max_frontier=4)
        st = tree.state()
        n = int(fx[f"{case}_n_nodes"][0])
        assert st["status"].tolist() == [0, 0]
        assert st["n_nodes"].tolist() == [n, n]
        for b in range(2):
            assert st["parents"][b, :n].tolist() == ints(f"{case}_parents")
            assert st["tokens"][b, :n].tolist() == ints(f"{case}_tokens")
            np.testing.assert_allclose(st["entropy"][b, :4], floats("entropy"), atol=1e-5)
            assert st["width"][b, :4].tolist() == ints("width")
        if case == "caseA":
            np.testing.assert_allclose(st["scores"][0, :n], floats("caseA_scores"), atol=1e-5)


@pytest.mark.parametrize("B,n_max,V,levels,top_k,max_new", [
    (3, 64, 1000, 6, 8, 16),       # one slice per row
    (2, 64, 4099, 6, 8, 16),       # V not a multiple of 4: scalar loads
    (4, 32, 20001, 5, 6, 12),      # three slices, ragged tail
    (2, 16, 24576, 4, 8, 8),       # whole slices, no tail
    (5, 64, 37, 6, 3, 64),         # tiny vocabulary, one level may add every candidate
    (1, 64, 128256, 6, 8, 16),     # the 128K vocabulary, 16 slices
    (3, 16, 1, 3, 8, 8),           # one token: every node has one child, score 0
    (2, 16, 5, 4, 8, 16),          # fewer tokens than top_k
])
def test_levels_match_oracle(B, n_max, V, levels, top_k, max_new):
    dev = require_gpu()
    wl = W.make_expand_workload(B, n_max, V, seed=V + B, n_levels=levels, top_k=top_k, max_new=max_new)
    st, near, rows = _grow_and_compare(wl, dev)
    assert np.all(st["status"] == 0)
    assert near <= max(1, B * levels // 4), f"{near} near-boundary request-levels"


@pytest.mark.parametrize("name", ["llama2_7b", "llama3_70b", "serving"])
def test_full_size_levels_match_oracle(name):
    """The vocabularies and batches of the verification workloads, with
    n_max = 64, depth 6, top_k 8 and 16 nodes per level."""
    dev = require_gpu()
    cfg = W.CONFIG_BY_NAME[name]
    B = min(cfg.B, 8)
    wl = W.make_expand_workload(B, 64, cfg.V, seed=cfg.seed, n_levels=6, top_k=8, max_new=16,
                                sigma_flat=cfg.sigma)
    st, near, rows = _grow_and_compare(wl, dev)
    assert np.all(st["status"] == 0)
    assert near <= max(1, B * 6 // 4)
    assert np.all(st["n_nodes"] <= 64)


def test_chain_for_peaked_rows_and_top_k_one():
    dev = require_gpu()
    rng = np.random.default_rng(11)
    V, n_max = 5000, 16
    rows = rng.standard_normal((2, n_max, V)).astype(np.float32)
    spikes = rng.integers(0, V, size=(2, n_max))
    for b in range(2):
        rows[b, np.arange(n_max), spikes[b]] += 40.0
    tree = DevTree(rows, [1, 2], dev, n_max)
    for _ in range(6):
        tree.level(8, 16, n_max, max_frontier=16)
    st = tree.state()
    assert st["n_nodes"].tolist() == [7, 7]
    for b in range(2):
        assert st["parents"][b, :7].tolist() == list(range(-1, 6))
        assert st["tokens"][b, 1:7].tolist() == spikes[b, :6].tolist()
    # top_k = 1 on flat rows: a greedy chain of argmax tokens
    flat = (3.0 * rng.standard_normal((1, n_max, V))).astype(np.float32)
    tree = DevTree(flat, [0], dev, n_max)
    for _ in range(5):
        tree.level(1, 16, n_max, max_frontier=16)
    st = tree.state()
    assert st["n_nodes"][0] == 6
    assert st["tokens"][0, 1:6].tolist() == [int(np.argmax(flat[0, f])) for f in range(5)]


def test_status_edges_and_budget():
    dev = require_gpu()
    V, n_max = 64, 8
    rng = np.random.default_rng(12)
    rows = rng.standard_normal((5, n_max, V)).astype(np.float32)
    tree = DevTree(rows, [0] * 5, dev, n_max)
    # request 0: invalid n_nodes; 1: level_start past n_nodes; 2: incoming
    # status; 3: frontier wider than max_frontier; 4: budget already reached
    tree.n_nodes[0] = 0
    tree.n_nodes[1], tree.level_start[1] = 2, 3
    tree.status[2] = 2
    tree.n_nodes[3], tree.level_start[3] = 5, 1
    tree.parents[3, 1:5] = torch.tensor([0, 0, 0, 0], dtype=torch.int32)
    tree.n_nodes[4], tree.level_start[4] = 4, 1
    tree.parents[4, 1:4] = torch.tensor([0, 0, 0], dtype=torch.int32)
    before = tree.state()
    tree.level(8, 8, 4, max_frontier=3)
    st = tree.state()
    assert st["status"].tolist() == [oracle.STATUS_BAD_TREE, oracle.STATUS_BAD_TREE, 2, oracle.STATUS_CAPACITY, 0]
    for b in range(4):
        assert st["n_nodes"][b] == before["n_nodes"][b]
        assert st["level_start"][b] == before["level_start"][b]
        assert st["parents"][b].tolist() == before["parents"][b].tolist()
    assert st["n_nodes"][4] == 4 and st["level_start"][4] == 4
    assert st["parents"][4].tolist() == before["parents"][4].tolist()


def test_workspace_reuse_optional_outputs_and_errors():
    dev = require_gpu()
    wl = W.make_expand_workload(3, 64, 3000, seed=9, n_levels=4)
    tree = DevTree(wl.draft_logits, wl.root_tokens, dev, 64)
    ws = tvb.new_expand_workspace(3, 16, 3000, dev)
    for _ in range(4):                       # one zero-filled workspace serves every level
        tvb.tree_expand(tree.logits, tree.parents, tree.tokens, tree.scores, tree.n_nodes, tree.level_start,
                        tree.status, top_k=8, max_new=16, budget=64, max_frontier=16, workspace=ws)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(ws[-3 * 4:])) == 0          # arrival counters back at zero
    ref = oracle.tree_build_dynamic(wl.draft_logits, wl.root_tokens, 4, 8, 16, 64)
    st = tree.state()
    for b in range(3):
        if ref["near_boundary"][b]:
            continue
        n = int(ref["n_nodes"][b])
        assert st["n_nodes"][b] == n
        assert st["parents"][b, :n].tolist() == ref["parents"][b, :n].tolist()
        assert st["tokens"][b, :n].tolist() == ref["tokens"][b, :n].tolist()
    with pytest.raises(tvb.TreeVerifyError):
        tvb.tree_expand(tree.logits, tree.parents, tree.tokens, tree.scores, tree.n_nodes, tree.level_start,
                        tree.status, top_k=9, max_new=16, budget=64)
    with pytest.raises(tvb.TreeVerifyError):
        tvb.tree_expand(tree.logits, tree.parents, tree.tokens, tree.scores, tree.n_nodes, tree.level_start,
                        tree.status, top_k=8, max_new=16, budget=65)
    with pytest.raises(tvb.TreeVerifyError):
        tvb.tree_expand(tree.logits, tree.parents, tree.tokens, tree.scores, tree.n_nodes, tree.level_start,
                        tree.status, top_k=8, max_new=16, budget=64, max_frontier=16, workspace=ws[:64])


def test_rows_with_many_equal_logits():
    """Logits rounded to a coarse grid (thousands of equal values per slice,
    more than the threshold filter keeps) and constant rows: the exact
    per-thread path and the lower-id-first tie rule."""
    dev = require_gpu()
    rng = np.random.default_rng(13)
    B, n_max, V = 3, 32, 20000
    rows = np.round(rng.standard_normal((B, n_max, V)) * 1.5).astype(np.float32)
    rows[0, :4] = 0.0                          # uniform rows: every token equally likely
    rows[1, 0, 5000:5003] = 9.0                # three equal spikes
    wl = W.ExpandWorkload(B=B, n_max=n_max, V=V, draft_logits=rows, kinds=np.zeros((B, n_max), np.int8),
                          root_tokens=np.zeros(B, np.int32), n_levels=4, top_k=8, max_new=10, budget=n_max)
    st, near, rows_read = _grow_and_compare(wl, dev)
    assert np.all(st["status"] == 0)
    assert st["tokens"][0, 1:9].tolist() == list(range(8))     # uniform root row: the 8 lowest ids


def test_large_batch():
    """520 requests (grid z beyond a few hundred) on a small vocabulary."""
    dev = require_gpu()
    wl = W.make_expand_workload(520, 16, 2048, seed=21, n_levels=3, top_k=4, max_new=6)
    st, near, rows = _grow_and_compare(wl, dev)
    assert np.all(st["status"] == 0)
    assert near <= 520 * 3 // 20
