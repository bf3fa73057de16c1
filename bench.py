#!/usr/bin/env python
"""Benchmark of the tree-verification step on GB300.

One step = the whole hot path over one batch of synthetic input:
tv_tree_build_mask -> tv_tree_verify_attn -> tv_tree_accept -> tv_kv_commit_path.
The default workload is the Llama-3-70B-shaped verify (batch 8, 64 query / 8
KV heads, head dim 128, prefixes 1024-8192 in shuffled 16-token pages, 64-node
trees of depth 4-6, rejection-sampling acceptance at T = 0.7 over 128256
logits, commit across 80 layers).

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and torch.cuda.synchronize(); CUDA events on the launching stream.  Each step
is one replay of a CUDA graph of the four calls; rotated copies of the inputs
(KV cache, queries, logits) make the data one step reads exceed 3x L2, so no
step finds the previous step's inputs in L2.  The accept+commit pair is timed
on its own over the same rotation.  Then each Llama-shaped workload's
attention is timed alone over at least --leg-seconds of back-to-back calls
(rotated caches > 3x L2) with the SM clock sampled during it; this config's
leg gives the roofline object.

--impl reference times the fp64 CPU oracle instead (bounded sample of the
same workload, attention rows spread over the host cores).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "tree-verify attention TB/s & % roofline; verified tree nodes/s; accept+commit µs"
L2_BYTES = 126 * 1024 * 1024


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="llama3_70b")
    ap.add_argument("--leg-seconds", type=float, default=2.0,
                    help="minimum timed seconds of each workload's attention leg (clocks sampled during it)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-attn", type=int, default=0,
                    help="only run this many eager tv_tree_verify_attn calls (for profiler captures)")
    ap.add_argument("--profile-attn-q4", type=int, default=0,
                    help="profiler capture mode: N eager tv_tree_verify_attn_q4 calls on the chosen config's cache "
                         "encoded in the 4-bit format, and exit")
    ap.add_argument("--profile-expand", type=int, default=0,
                    help="profiler capture mode: build N trees (6 levels each) with tv_tree_expand and exit")
    ap.add_argument("--profile-accept", type=int, default=0,
                    help="profiler capture mode: N tree_accept calls on the chosen config (its greedy or sampling "
                         "mode) and exit")
    ap.add_argument("--profile-step", type=int, default=0,
                    help="profiler capture mode: N eager steps (mask, attention, accept, commit) and exit")
    ap.add_argument("--profile-quant", type=int, default=0,
                    help="profiler capture mode: N 4-bit encodings of the chosen config's K cache layer and exit")
    ap.add_argument("--breakdown", action="store_true",
                    help="print per-call times of every kernel on each verification workload (CUDA graphs of ten "
                         "calls, L2-warm) and the 6-level expansion time, one JSON line per workload, and exit")
    ap.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--oracle-accept", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args()


# ------------------------------------------------------------------ oracle leg
def oracle_sample_plan(cfg_name):
    """Bounded sample of the workload for the CPU oracle."""
    from eagle_speculative_decoding_attn_gb300 import workloads as W
    cfg = W.CONFIG_BY_NAME[cfg_name]
    if cfg_name in ("tiny", "llama2_7b"):
        return dict(B=cfg.B, heads=cfg.Hq, desc="the full step (all requests, all heads)")
    heads = max(1, cfg.Hq // 16)
    return dict(B=1, heads=heads,
                desc=f"one request drawn from the same generator, {heads} of {cfg.Hq} query heads for "
                     f"attention, full accept/commit; scaled to the full batch by attention key counts")


_POOL_W = None


def _pool_init(cfg_name, B):
    """Worker set-up for the all-cores oracle timing: the same seeded sample."""
    global _POOL_W
    from eagle_speculative_decoding_attn_gb300 import workloads as W
    _POOL_W = W.make_workload(cfg_name, B=B)


def _pool_attn(rows):
    """The oracle's attention on a share of the sample's (request, node, head) rows."""
    import oracle
    w = _POOL_W
    oracle.tree_verify_attn(w.q_bits, w.k_bits, w.v_bits, w.page_table, w.prefix_len, w.n_nodes, w.parents,
                            w.scale, rows=rows)
    return len(rows)


def run_oracle_sample(cfg_name):
    """Time the oracle (as it stands) on the bounded sample; returns seconds
    per full step (scaled) and the sample description.  The attention part is
    also timed with its rows spread over every host core (spawned worker
    processes, one thread each); mask, accept and commit stay single-thread."""
    import numpy as np
    import oracle
    from eagle_speculative_decoding_attn_gb300 import workloads as W
    plan = oracle_sample_plan(cfg_name)
    cfg = W.CONFIG_BY_NAME[cfg_name]
    w = W.make_workload(cfg_name, B=plan["B"])
    full = W.make_workload(cfg_name, with_logits=False) if plan["B"] != cfg.B else w
    rows = [(b, i, h) for b in range(w.B) for i in range(int(w.n_nodes[b])) for h in range(plan["heads"])]
    t0 = time.perf_counter()
    oracle.tree_build_mask(w.parents, w.n_nodes)
    t1 = time.perf_counter()
    oracle.tree_verify_attn(w.q_bits, w.k_bits, w.v_bits, w.page_table, w.prefix_len, w.n_nodes, w.parents,
                            w.scale, rows=rows)
    t2 = time.perf_counter()
    if w.temperature > 0:
        acc = oracle.tree_accept_sampling(w.target_logits, w.draft_logits, w.tokens, w.parents, w.n_nodes,
                                          w.temperature, w.u_accept, w.u_sample)
    else:
        acc = oracle.tree_accept_greedy(w.target_logits, w.tokens, w.parents, w.n_nodes)
    t3 = time.perf_counter()
    oracle.kv_commit_path(w.k_bits[None], w.v_bits[None], w.page_table, w.prefix_len, w.n_nodes,
                          acc["accept_len"], acc["path_nodes"])
    t4 = time.perf_counter()
    tot_keys = float(np.sum((full.prefix_len.astype(np.float64) + full.n_nodes) * full.n_nodes) * full.Hq)
    smp_keys = float(sum(int(w.prefix_len[b]) + int(w.n_nodes[b]) for (b, i, h) in rows))
    f_attn = tot_keys / max(smp_keys, 1.0)
    f_req = full.B / w.B
    t_rest = (t1 - t0) * f_req + (t3 - t2) * f_req + (t4 - t3) * f_req * cfg.n_layers_commit
    t_step = t_rest + (t2 - t1) * f_attn
    # the attention rows over every core
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    t_par = t2 - t1
    if cores > 1:
        # whole nodes per worker: the oracle gathers a node's key sequence once for all its heads
        nodes = sorted({(b, i) for (b, i, h) in rows})
        share = {n: k % cores for k, n in enumerate(nodes)}
        chunks = [[r for r in rows if share[(r[0], r[1])] == k] for k in range(cores)]
        chunks = [c for c in chunks if c]
        with mp.get_context("spawn").Pool(len(chunks), initializer=_pool_init, initargs=(cfg_name, plan["B"])) as pool:
            pool.map(_pool_attn, [c[:1] for c in chunks])        # workers ready, code warm
            tp = time.perf_counter()
            pool.map(_pool_attn, chunks)
            t_par = time.perf_counter() - tp
    return dict(seconds_per_step=t_step, nodes=float(np.sum(full.n_nodes)), cpu_seconds=t4 - t0,
                desc=plan["desc"], cores=cores if cores > 1 else 1,
                seconds_per_step_all_cores=t_rest + t_par * f_attn)


def run_oracle_accept(cfg_name):
    """The oracle's acceptance of the whole batch (greedy or sampling, as the
    workload says): accepted lengths and near-boundary flags per request."""
    import numpy as np
    import oracle
    from eagle_speculative_decoding_attn_gb300 import workloads as W
    w = W.make_workload(cfg_name)
    if w.temperature > 0:
        r = oracle.tree_accept_sampling(w.target_logits, w.draft_logits, w.tokens, w.parents, w.n_nodes,
                                        w.temperature, w.u_accept, w.u_sample)
        nb = np.asarray(r["near_boundary"], dtype=bool)
    else:
        r = oracle.tree_accept_greedy(w.target_logits, w.tokens, w.parents, w.n_nodes)
        nb = np.zeros(w.B, dtype=bool)
    return {"accept_len": [int(x) for x in r["accept_len"]], "near_boundary": nb.tolist()}


def oracle_accept_subprocess(cfg_name):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-accept", "--config", cfg_name],
                       env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def oracle_leg_subprocess(cfg_name):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               NUMEXPR_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-sample", "--config", cfg_name],
                       env=env, capture_output=True, text=True, timeout=1200)
    if r.returncode != 0:
        raise RuntimeError(r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline_obj(res):
    return {"value": res["nodes"] / res["seconds_per_step_all_cores"], "unit": "nodes/s", "cores": res["cores"],
            "kind": "oracle",
            "single_thread": {"value": res["nodes"] / res["seconds_per_step"], "cores": 1},
            "sample": f"{res['desc']}; {res['cpu_seconds']:.1f} s of single-thread CPU work, "
                      f"{res['seconds_per_step']:.1f} s per full step on one core, "
                      f"{res['seconds_per_step_all_cores']:.2f} s with the attention rows spread over "
                      f"{res['cores']} cores (one process each)"}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, cuda_index):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        self.gpu = ids[cuda_index] if cuda_index < len(ids) and ids[cuda_index].isdigit() else str(cuda_index)
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [[c.strip() for c in r.split(",")] for r in out.strip().splitlines() if r.count(",") >= 8]
        num = lambda x: x.replace(".", "", 1).isdigit()
        sm = sorted(float(r[1]) for r in rows if num(r[1]))
        mx = [float(r[2]) for r in rows if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for k, nm in enumerate(names):
                if r[5 + k] == "Active":
                    reasons.add(nm)
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def workload_config(cfg, world):
    """The `config` keys naming the workload, the same on both arms' lines."""
    return {"workload": f"{cfg.name}: B={cfg.B}, Hq={cfg.Hq}, Hkv={cfg.Hkv}, D={cfg.D}, prefix={cfg.prefix}, "
                        f"nodes={cfg.n_nodes}, V={cfg.V}, T={cfg.temperature}, commit layers={cfg.n_layers_commit}",
            "global_batch": cfg.B * world, "parallelism": f"replicas x{world}"}


def packed_views(buf, specs):
    """Views of a flat uint8 tensor as the (name, dtype, shape) arrays of `specs`,
    each starting on a 256-byte boundary; returns ({name: view}, total bytes).
    With buf None only the size is computed."""
    import numpy as np
    views, off = {}, 0
    for name, dtype, shape in specs:
        n = int(np.prod(shape)) * dtype.itemsize
        if buf is not None:
            views[name] = buf[off:off + n].view(dtype).view(shape)
        off = (off + n + 255) // 256 * 256
    return views, off


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------ GPU leg
def reduce_over_ranks(times, work, device):
    """Whole-job figures of a replicated run: each timing is the maximum over
    the ranks and each work count the sum (one all-reduce each); unchanged on a
    single rank.  `device` is where the reduction tensors live (the GPU for
    NCCL, the CPU for gloo)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(x) for x in times], [float(x) for x in work]
    t = torch.tensor(times, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    n = torch.tensor(work, dtype=torch.float64, device=device)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return [float(x) for x in t.tolist()], [float(x) for x in n.tolist()]


def profile_attn(args, W, tvb, dev):
    """A small self-contained command for profiler captures: mask once, then
    N eager attention calls on the chosen config."""
    import numpy as np
    import torch
    w = W.make_workload(args.config, with_logits=False)
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    bf = lambda bits: g(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    parents, n_nodes = g(w.parents), g(w.n_nodes)
    q, k, v = bf(w.q_bits), bf(w.k_bits), bf(w.v_bits)
    pt, L = g(w.page_table), g(w.prefix_len)
    anc, depth, status = tvb.tree_build_mask(parents, n_nodes)
    ws = tvb.new_attn_workspace(w.B, w.n_max, w.Hq, w.Hkv, w.D, dev)
    if args.profile_attn_q4:
        kc, kp = tvb.kv_quantize_q4(k)
        vc, vp = tvb.kv_quantize_q4(v)
        del k, v
        for _ in range(args.profile_attn_q4):
            tvb.tree_verify_attn_q4(q, kc, kp, vc, vp, pt, L, n_nodes, anc, w.scale, status, workspace=ws)
        torch.cuda.synchronize()
        print(json.dumps({"profile_attn_q4": args.config, "calls": args.profile_attn_q4,
                          "status": status.cpu().numpy().tolist(), "attn_bytes_q4": w.attn_bytes_q4()}))
        return
    for _ in range(args.profile_attn):
        tvb.tree_verify_attn(q, k, v, pt, L, n_nodes, anc, w.scale, status, workspace=ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile_attn": args.config, "calls": args.profile_attn,
                      "status": status.cpu().numpy().tolist(), "kv_bytes": int(w.k_bits.nbytes * 2)}))


def time_expand(args, W, tvb, torch, np, dev, stream, B, n_max, V, cfg):
    """Dynamic tree construction on its own: `levels` launches of
    tv_tree_expand per tree over seeded drafter rows of the workload's batch and
    vocabulary, each tree from a fresh root; rotated logits copies keep the
    rows out of L2.  The state reset (one device copy per tree) is timed
    separately and subtracted."""
    levels, top_k, max_new = 6, 8, 16
    ew = W.make_expand_workload(B, n_max, V, seed=cfg.seed, n_levels=levels, top_k=top_k, max_new=max_new,
                                sigma_flat=cfg.sigma)
    Bn = B * n_max
    init = torch.zeros(4 * Bn + 3 * B, dtype=torch.int32)
    init[0:Bn] = -1                                                  # parents
    init[Bn:2 * Bn].view(B, n_max)[:, 0] = torch.from_numpy(ew.root_tokens)
    init[4 * Bn:4 * Bn + B] = 1                                      # n_nodes
    init = init.to(dev)
    RE = min(64, max(1, math.ceil(3 * L2_BYTES / ew.draft_logits.nbytes)))
    logits0 = torch.from_numpy(ew.draft_logits).to(dev)
    copies = []
    for _ in range(RE):
        st = init.clone()
        copies.append(dict(logits=logits0.clone(), state=st, parents=st[0:Bn].view(B, n_max),
                           tokens=st[Bn:2 * Bn].view(B, n_max), scores=st[2 * Bn:3 * Bn].view(torch.float32).view(B, n_max),
                           width=st[3 * Bn:4 * Bn].view(B, n_max), n_nodes=st[4 * Bn:4 * Bn + B],
                           level_start=st[4 * Bn + B:4 * Bn + 2 * B], status=st[4 * Bn + 2 * B:],
                           ws=tvb.new_expand_workspace(B, max_new, V, dev)))
    del logits0

    def build(ec):
        for _ in range(levels):
            tvb.tree_expand(ec["logits"], ec["parents"], ec["tokens"], ec["scores"], ec["n_nodes"], ec["level_start"],
                            ec["status"], top_k=top_k, max_new=max_new, budget=n_max, max_frontier=max_new,
                            width=ec["width"], workspace=ec["ws"])

    for ec in copies:
        ec["state"].copy_(init)
        build(ec)
    torch.cuda.synchronize()
    side = torch.cuda.Stream(dev)
    g_all, g_rst = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g_all, stream=side):
            for ec in copies:
                ec["state"].copy_(init)
                build(ec)
        with torch.cuda.graph(g_rst, stream=side):
            for ec in copies:
                ec["state"].copy_(init)
    torch.cuda.synchronize()
    reps = max(3, min(50, args.steps // RE + 1))
    times = []
    for gph in (g_all, g_rst):
        gph.replay()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(reps):
            gph.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        times.append(t0.elapsed_time(t1) * 1000.0 / (reps * RE))
    g_all.replay()                      # leave every copy holding a finished tree
    torch.cuda.synchronize()
    ec = copies[0]
    rows_read = int((ec["width"] > 0).sum().item())
    return {"us_per_tree": times[0] - times[1], "reset_us": times[1], "levels": levels, "top_k": top_k,
            "max_new_per_level": max_new, "budget": n_max, "rows_read": rows_read,
            "nodes": int(ec["n_nodes"].sum().item()), "bytes": rows_read * V * 4,
            "status_ok": bool((ec["status"] == 0).all().item()),
            "l2": f"{RE} rotated logits copies ({RE * ew.draft_logits.nbytes / 1e6:.0f} MB)"}


def attn_roofline(abytes, aflops, us, hbm, tf_burst, traffic=None):
    """Roofline object of one attention timing: the slower of the algorithmic
    bytes at the measured HBM bandwidth and the FLOPs at the measured bf16 peak."""
    t_hbm = abytes / (hbm * 1e9)
    t_tc = aflops / (tf_burst * 1e12)
    s = us * 1e-6
    if t_hbm >= t_tc:
        bound, achieved, peak, unit = "hbm", abytes / s / 1e9, hbm, "GB/s"
    else:
        bound, achieved, peak, unit = "tensor", aflops / s / 1e12, tf_burst, "TFLOP/s"
    return {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
            "traffic": traffic, "bound_us": max(t_hbm, t_tc) * 1e6}


def load_traffic(name, kind="attn"):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload (profiles/traffic_<kind>_<name>.json), or None."""
    path = os.path.join(ROOT, "profiles", f"traffic_{kind}_{name}.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        return json.load(f).get("dram_bytes_per_launch")


def attn_legs(W, tvb, dev, local_rank, names, min_seconds=2.0, q4_seconds=1.0):
    """Each workload's attention on its own, over at least `min_seconds` of
    back-to-back calls: one CUDA graph holds one call per rotated copy of the
    cache (copies enough to exceed 3x L2, so no call finds its K/V in L2) and is
    replayed; CUDA events on the launching stream time the whole region and the
    SM clock is sampled during it.  Then the same over the cache encoded in the
    4-bit format (tv_tree_verify_attn_q4)."""
    import numpy as np
    import torch
    hbm, tf_burst, _ = load_peaks()
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    bf = lambda b: g(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)
    stream = torch.cuda.current_stream(dev)
    legs = {}

    def timed(calls, seconds):
        side = torch.cuda.Stream(dev)
        gr = torch.cuda.CUDAGraph()
        for c in calls:
            c()
        torch.cuda.synchronize()
        with torch.cuda.stream(side):
            with torch.cuda.graph(gr, stream=side):
                for c in calls:
                    c()
        torch.cuda.synchronize()
        for _ in range(3):
            gr.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(3):
            gr.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        est = e0.elapsed_time(e1) / 3 / 1000.0
        n = max(3, int(math.ceil(seconds / max(est, 1e-6))))
        clocks = ClockSampler(local_rank)
        clocks.start()
        time.sleep(0.3)
        e0.record(stream)
        for _ in range(n):
            gr.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        clk = clocks.stop()
        ms = e0.elapsed_time(e1)
        return ms * 1000.0 / (n * len(calls)), ms / 1000.0, n * len(calls), clk

    for name in names:
        w = W.make_workload(name, with_logits=False)
        per = w.k_bits.nbytes * 2 + w.q_bits.nbytes
        R = min(16, max(1, math.ceil(3 * L2_BYTES / per)))
        pt, L, n_nodes, parents = g(w.page_table), g(w.prefix_len), g(w.n_nodes), g(w.parents)
        q = bf(w.q_bits)
        kv = [(bf(w.k_bits), bf(w.v_bits)) for _ in range(R)]
        anc, _, st = tvb.tree_build_mask(parents, n_nodes)
        ws = tvb.new_attn_workspace(w.B, w.n_max, w.Hq, w.Hkv, w.D, dev)
        out = torch.empty_like(q)
        lse = torch.empty((w.B, w.n_max, w.Hq), dtype=torch.float32, device=dev)
        calls = [lambda k=k, v=v: tvb.tree_verify_attn(q, k, v, pt, L, n_nodes, anc, w.scale, st, out=out, lse=lse,
                                                       workspace=ws) for (k, v) in kv]
        us, secs, launches, clk = timed(calls, min_seconds)
        abytes, aflops = w.attn_bytes(), w.attn_flops()
        leg = {"us": us, "timed_s": secs, "launches": launches, "rotated_copies": R,
               "tbps": abytes / us / 1e6, "nodes_per_s": float(np.sum(w.n_nodes)) / (us * 1e-6),
               "status_ok": bool((st == 0).all().item()),
               "roofline": attn_roofline(abytes, aflops, us, hbm, tf_burst, load_traffic(name)),
               "algorithmic": {"bytes": abytes, "flops": aflops, "exps": aflops // (4 * w.D)},
               "clocks": clk}
        if q4_seconds > 0:
            enc = [tvb.kv_quantize_q4(k) + tvb.kv_quantize_q4(v) for (k, v) in kv]
            del kv
            qcalls = [lambda c=c: tvb.tree_verify_attn_q4(q, *c, pt, L, n_nodes, anc, w.scale, st, out=out, lse=lse,
                                                          workspace=ws) for c in enc]
            qus, qsecs, qlaunches, qclk = timed(qcalls, q4_seconds)
            qbytes = w.attn_bytes_q4()
            leg["q4"] = {"us": qus, "timed_s": qsecs, "launches": qlaunches, "tbps": qbytes / qus / 1e6,
                         "status_ok": bool((st == 0).all().item()),
                         "vs_bf16": us / qus,
                         "roofline": attn_roofline(qbytes, aflops, qus, hbm, tf_burst, load_traffic(name, "attn_q4")),
                         "bytes": qbytes, "clocks": qclk}
            del enc
        else:
            del kv
        legs[name] = leg
        torch.cuda.empty_cache()
    return legs


def profile_expand(args, W, tvb, dev):
    """A small self-contained command for profiler captures: N eager tree
    builds of 6 levels of dynamic expansion on the chosen config's batch and
    vocabulary."""
    import numpy as np
    import torch
    cfg = W.CONFIG_BY_NAME[args.config]
    B, V, n_max = cfg.B, cfg.V, 64
    ew = W.make_expand_workload(B, n_max, V, seed=cfg.seed, n_levels=6, sigma_flat=cfg.sigma)
    logits = torch.from_numpy(ew.draft_logits).to(dev)
    ws = tvb.new_expand_workspace(B, 16, V, dev)
    for _ in range(args.profile_expand):
        par = torch.full((B, n_max), -1, dtype=torch.int32, device=dev)
        tok = torch.zeros((B, n_max), dtype=torch.int32, device=dev)
        tok[:, 0] = torch.from_numpy(ew.root_tokens).to(dev)
        sc = torch.zeros((B, n_max), dtype=torch.float32, device=dev)
        n = torch.ones(B, dtype=torch.int32, device=dev)
        ls = torch.zeros(B, dtype=torch.int32, device=dev)
        st = torch.zeros(B, dtype=torch.int32, device=dev)
        for _ in range(6):
            tvb.tree_expand(logits, par, tok, sc, n, ls, st, top_k=8, max_new=16, budget=n_max, max_frontier=16,
                            workspace=ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile_expand": args.config, "trees": args.profile_expand,
                      "n_nodes": n.cpu().numpy().tolist(), "status": st.cpu().numpy().tolist()}))


def breakdown(args, W, tvb, dev):
    """Per-call cost of each kernel inside CUDA graphs of ten calls (inputs
    L2-warm) on the four Llama-shaped workloads, and six levels of tree
    expansion on each workload's batch and vocabulary."""
    import numpy as np
    import torch
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    bf = lambda b: g(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)

    def gtime(fn, n=10, reps=200):
        fn()
        torch.cuda.synchronize()
        s = torch.cuda.Stream(dev)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(gr, stream=s):
                for _ in range(n):
                    fn()
        torch.cuda.synchronize()
        for _ in range(3):
            gr.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            gr.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1000 / (reps * n)

    hbm, tf_burst, _ = load_peaks()
    for name in ("llama2_7b", "llama3_70b", "serving", "long"):
        w = W.make_workload(name)
        cfg = W.CONFIG_BY_NAME[name]
        sampling = w.temperature > 0
        parents, n_nodes, L, pt, tokens = g(w.parents), g(w.n_nodes), g(w.prefix_len), g(w.page_table), g(w.tokens)
        target = g(w.target_logits)
        draft = g(w.draft_logits) if sampling else None
        ua = g(w.u_accept) if sampling else None
        us = g(w.u_sample) if sampling else None
        layers = cfg.n_layers_commit
        k = bf(w.k_bits).unsqueeze(0).repeat(layers, 1, 1, 1, 1).contiguous()
        v = bf(w.v_bits).unsqueeze(0).repeat(layers, 1, 1, 1, 1).contiguous()
        q = bf(w.q_bits)
        anc, depth, status = tvb.tree_build_mask(parents, n_nodes)
        ws = tvb.new_attn_workspace(w.B, w.n_max, w.Hq, w.Hkv, w.D, dev)
        aws = tvb.new_accept_workspace(w.B, w.n_max, w.V, dev)
        out = torch.empty_like(q)
        lse = torch.empty((w.B, w.n_max, w.Hq), dtype=torch.float32, device=dev)
        t_mask = gtime(lambda: tvb.tree_build_mask(parents, n_nodes, anc_mask=anc, depth=depth, status=status))
        t_attn = gtime(lambda: tvb.tree_verify_attn(q, k[0], v[0], pt, L, n_nodes, anc, w.scale, status, out=out,
                                                    lse=lse, workspace=ws))
        # the same attention over the layer's cache encoded in the 4-bit format
        kc, kp = tvb.kv_quantize_q4(k[0])
        vc, vp = tvb.kv_quantize_q4(v[0])
        t_attn_q4 = gtime(lambda: tvb.tree_verify_attn_q4(q, kc, kp, vc, vp, pt, L, n_nodes, anc, w.scale, status,
                                                          out=out, lse=lse, workspace=ws))
        del kc, kp, vc, vp
        acc = tvb.tree_accept(target, draft, tokens, parents, n_nodes, anc, depth, w.temperature, ua, us, status,
                              workspace=aws)
        t_acc = gtime(lambda: tvb.tree_accept(target, draft, tokens, parents, n_nodes, anc, depth, w.temperature, ua,
                                              us, status, outputs=acc, workspace=aws))
        t_acc_wor = None
        if sampling:  # the sibling rule for trees drafted without replacement, same inputs
            t_acc_wor = gtime(lambda: tvb.tree_accept(target, draft, tokens, parents, n_nodes, anc, depth,
                                                      w.temperature, ua, us, status, outputs=acc, workspace=aws,
                                                      without_replacement=True))
            tvb.tree_accept(target, draft, tokens, parents, n_nodes, anc, depth, w.temperature, ua, us, status,
                            outputs=acc, workspace=aws)
        com = tvb.kv_commit_path(k, v, pt, L, n_nodes, acc[0], acc[1], status)
        t_com = gtime(lambda: tvb.kv_commit_path(k, v, pt, L, n_nodes, acc[0], acc[1], status, outputs=com))
        # release of the rejected pages: page table and counts restored by a device copy before
        # each call; the copies alone are timed too and subtracted
        pt0, rc0 = pt.clone(), torch.ones(w.num_pages, dtype=torch.int32, device=dev)
        ptw, rcw = pt.clone(), rc0.clone()
        fl = torch.empty(w.B * 8, dtype=torch.int32, device=dev)
        fc = torch.zeros(1, dtype=torch.int32, device=dev)
        pst = torch.zeros_like(status)

        def restore():
            ptw.copy_(pt0)
            rcw.copy_(rc0)
            fc.zero_()
        t_prune = gtime(lambda: (restore(), tvb.kv_prune_pages(ptw, rcw, L, n_nodes, com[1], pst, free_list=fl,
                                                                 free_count=fc))) - gtime(restore)
        freed = int(fc.item())
        ok = bool((status == 0).all().item())
        # 4-bit encoding of one layer's K cache (every page of the batch)
        qc, qp = tvb.kv_quantize_q4(k[0])
        t_q4 = gtime(lambda: tvb.kv_quantize_q4(k[0], codes=qc, params=qp))
        q4_bytes = k[0].numel() * 2 + qc.numel() + qp.numel() * 2
        del qc, qp
        del k, v, target, draft
        torch.cuda.empty_cache()
        # six levels of expansion from a fresh root, the reset outside the graph
        ew = W.make_expand_workload(w.B, 64, w.V, seed=cfg.seed, n_levels=6, sigma_flat=cfg.sigma)
        logits = g(ew.draft_logits)
        st = [torch.full((w.B, 64), -1, dtype=torch.int32, device=dev),
              torch.zeros((w.B, 64), dtype=torch.int32, device=dev),
              torch.zeros((w.B, 64), dtype=torch.float32, device=dev), torch.ones(w.B, dtype=torch.int32, device=dev),
              torch.zeros(w.B, dtype=torch.int32, device=dev), torch.zeros(w.B, dtype=torch.int32, device=dev)]
        st[1][:, 0] = g(ew.root_tokens)
        wd = torch.zeros((w.B, 64), dtype=torch.int32, device=dev)
        init = [x.clone() for x in st]
        xws = tvb.new_expand_workspace(w.B, 16, w.V, dev)

        def levels():
            for _ in range(6):
                tvb.tree_expand(logits, *st[:5], st[5], top_k=8, max_new=16, budget=64, max_frontier=16, width=wd,
                                workspace=xws)
        levels()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        sx = torch.cuda.Stream(dev)
        with torch.cuda.stream(sx):
            with torch.cuda.graph(gr, stream=sx):
                levels()
        ts = []
        for _ in range(12):
            for a, b in zip(st, init):
                a.copy_(b)
            wd.zero_()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            gr.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1000)
        t_exp = float(np.median(ts[2:]))
        rows = int((wd > 0).sum().item())
        ok = ok and bool((st[5] == 0).all().item())
        del logits
        torch.cuda.empty_cache()
        abytes, aflops = w.attn_bytes(), w.attn_flops()
        t_roof = max(abytes / (hbm * 1e3), aflops / (tf_burst * 1e6))
        qbytes = w.attn_bytes_q4()
        t_roof_q4 = max(qbytes / (hbm * 1e3), aflops / (tf_burst * 1e6))
        print(json.dumps({
            "workload": name, "status_ok": ok, "us_per_call": {
                "mask": t_mask, "attn": t_attn, "accept": t_acc, "accept_siblings_without_replacement": t_acc_wor,
                "commit": t_com, "prune_pages": t_prune},
            "pages_freed": freed,
            "kv_quantize_q4_one_layer_k": {"us": t_q4, "bytes": q4_bytes, "tbps": q4_bytes / t_q4 / 1e6},
            "attn_roofline_us": t_roof, "attn_bound": "hbm" if abytes / hbm >= aflops / tf_burst / 1e3 else "tensor",
            "attn_roofline_frac": t_roof / t_attn,
            "attn_q4": {"us": t_attn_q4, "bytes": qbytes, "roofline_us": t_roof_q4,
                        "bound": "hbm" if qbytes / hbm >= aflops / tf_burst / 1e3 else "tensor",
                        "roofline_frac": t_roof_q4 / t_attn_q4},
            "accept_mode": "sampling" if sampling else "greedy",
            "commit_layers": layers,
            "expand_6_levels": {"us": t_exp, "rows_read": rows, "bytes": rows * w.V * 4,
                                "tbps": rows * w.V * 4 / t_exp / 1e6}}), flush=True)


def profile_accept(args, W, tvb, dev):
    """A small self-contained command for profiler captures: N acceptance
    calls on the chosen config's tree and logits."""
    import numpy as np
    import torch
    w = W.make_workload(args.config)
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    sampling = w.temperature > 0
    parents, n_nodes, tokens = g(w.parents), g(w.n_nodes), g(w.tokens)
    target = g(w.target_logits)
    draft = g(w.draft_logits) if sampling else None
    ua = g(w.u_accept) if sampling else None
    us = g(w.u_sample) if sampling else None
    anc, depth, status = tvb.tree_build_mask(parents, n_nodes)
    aws = tvb.new_accept_workspace(w.B, w.n_max, w.V, dev)
    for _ in range(args.profile_accept):
        acc = tvb.tree_accept(target, draft, tokens, parents, n_nodes, anc, depth, w.temperature, ua, us, status,
                              workspace=aws)
    torch.cuda.synchronize()
    print(json.dumps({"profile_accept": args.config, "calls": args.profile_accept,
                      "mode": "sampling" if sampling else "greedy", "accept_len": acc[0].cpu().numpy().tolist(),
                      "status": status.cpu().numpy().tolist()}))


def profile_step(args, W, tvb, dev):
    """A small self-contained command for profiler launch lists: N eager steps
    (mask, attention, accept, commit over the config's layers) on the chosen
    config."""
    import numpy as np
    import torch
    cfg = W.CONFIG_BY_NAME[args.config]
    w = W.make_workload(args.config)
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    bf = lambda b: g(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)
    sampling = w.temperature > 0
    parents, n_nodes, tokens, L, pt = g(w.parents), g(w.n_nodes), g(w.tokens), g(w.prefix_len), g(w.page_table)
    target = g(w.target_logits)
    draft = g(w.draft_logits) if sampling else None
    ua = g(w.u_accept) if sampling else None
    us = g(w.u_sample) if sampling else None
    q = bf(w.q_bits)
    k = bf(w.k_bits).unsqueeze(0).repeat(cfg.n_layers_commit, 1, 1, 1, 1).contiguous()
    v = bf(w.v_bits).unsqueeze(0).repeat(cfg.n_layers_commit, 1, 1, 1, 1).contiguous()
    ws = tvb.new_attn_workspace(w.B, w.n_max, w.Hq, w.Hkv, w.D, dev)
    aws = tvb.new_accept_workspace(w.B, w.n_max, w.V, dev)
    for _ in range(args.profile_step):
        anc, depth, status = tvb.tree_build_mask(parents, n_nodes)
        tvb.tree_verify_attn(q, k[0], v[0], pt, L, n_nodes, anc, w.scale, status, workspace=ws)
        acc = tvb.tree_accept(target, draft, tokens, parents, n_nodes, anc, depth, w.temperature, ua, us, status,
                              workspace=aws)
        tvb.kv_commit_path(k, v, pt, L, n_nodes, acc[0], acc[1], status)
    torch.cuda.synchronize()
    print(json.dumps({"profile_step": args.config, "steps": args.profile_step,
                      "status": status.cpu().numpy().tolist()}))


def profile_quant(args, W, tvb, dev):
    """A small self-contained command for profiler captures: N 4-bit
    encodings of the chosen config's K cache (one layer)."""
    import numpy as np
    import torch
    w = W.make_workload(args.config, with_logits=False)
    k = torch.from_numpy(np.ascontiguousarray(w.k_bits).view(np.int16)).to(dev).view(torch.bfloat16)
    codes, params = tvb.kv_quantize_q4(k)
    for _ in range(args.profile_quant):
        tvb.kv_quantize_q4(k, codes=codes, params=params)
    torch.cuda.synchronize()
    print(json.dumps({"profile_quant": args.config, "calls": args.profile_quant,
                      "bytes_per_call": int(k.numel() * 2 + codes.numel() + params.numel() * 2)}))


def main():
    args = parse_args()
    if args.oracle_sample:
        print(json.dumps(run_oracle_sample(args.config)))
        return
    if args.oracle_accept:
        print(json.dumps(run_oracle_accept(args.config)))
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import numpy as np
    import torch
    import torch.distributed as dist
    from eagle_speculative_decoding_attn_gb300 import build as tvbuild
    from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
    from eagle_speculative_decoding_attn_gb300 import workloads as W

    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0:
        tvbuild.build()
    if world > 1:
        dist.barrier()
    tvb.load_library()
    if args.profile_attn or args.profile_attn_q4:
        return profile_attn(args, W, tvb, dev)
    if args.profile_expand:
        return profile_expand(args, W, tvb, dev)
    if args.breakdown:
        return breakdown(args, W, tvb, dev)
    if args.profile_accept:
        return profile_accept(args, W, tvb, dev)
    if args.profile_quant:
        return profile_quant(args, W, tvb, dev)
    if args.profile_step:
        return profile_step(args, W, tvb, dev)

    cfg = W.CONFIG_BY_NAME[args.config]
    w = W.make_workload(cfg)
    B, n_max, Hq, Hkv, D, V = w.B, w.n_max, w.Hq, w.Hkv, w.D, w.V
    sampling = w.temperature > 0
    layers = cfg.n_layers_commit
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    bf = lambda bits: g(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

    # bytes one step reads: layer-0 KV (attention), queries, logits
    per_copy = w.k_bits.nbytes * 2 + w.q_bits.nbytes + w.target_logits.nbytes * (2 if sampling else 1)
    R = min(16, max(1, math.ceil(3 * L2_BYTES / per_copy)))

    shared = dict(parents=g(w.parents), n_nodes=g(w.n_nodes), prefix_len=g(w.prefix_len),
                  page_table=g(w.page_table), tokens=g(w.tokens), u_accept=g(w.u_accept), u_sample=g(w.u_sample))
    k0, v0, q0, t0 = bf(w.k_bits), bf(w.v_bits), bf(w.q_bits), g(w.target_logits)
    d0 = g(w.draft_logits) if sampling else None
    # the step's results (accept and commit outputs) in one buffer per copy, so that
    # one device-to-host copy reads them back
    res_specs = [("accept_len", torch.int32, (B,)), ("path_nodes", torch.int32, (B, n_max)),
                 ("out_tokens", torch.int32, (B, n_max + 1)), ("slots", torch.int64, (B, n_max)),
                 ("new_len", torch.int32, (B,))]
    _, res_bytes = packed_views(None, res_specs)
    copies = []
    for _ in range(R):
        copies.append(dict(
            k=k0.unsqueeze(0).repeat(layers, 1, 1, 1, 1).contiguous(),
            v=v0.unsqueeze(0).repeat(layers, 1, 1, 1, 1).contiguous(),
            q=q0.clone(), target=t0.clone(), draft=d0.clone() if sampling else None,
            ws=tvb.new_attn_workspace(B, n_max, Hq, Hkv, D, dev),
            aws=tvb.new_accept_workspace(B, n_max, V, dev),
            anc=torch.empty((B, n_max), dtype=torch.int64, device=dev),
            depth=torch.empty((B, n_max), dtype=torch.int32, device=dev),
            status=torch.empty((B,), dtype=torch.int32, device=dev),
            out=torch.empty_like(q0), lse=torch.empty((B, n_max, Hq), dtype=torch.float32, device=dev),
            res=torch.empty(res_bytes, dtype=torch.uint8, device=dev)))
        rv, _ = packed_views(copies[-1]["res"], res_specs)
        copies[-1]["acc"] = (rv["accept_len"], rv["path_nodes"], rv["out_tokens"])
        copies[-1]["com"] = (rv["slots"], rv["new_len"])
    del k0, v0

    def mask_call(cp):
        tvb.tree_build_mask(shared["parents"], shared["n_nodes"], anc_mask=cp["anc"], depth=cp["depth"],
                            status=cp["status"])

    def attn_call(cp):
        tvb.tree_verify_attn(cp["q"], cp["k"][0], cp["v"][0], shared["page_table"], shared["prefix_len"],
                             shared["n_nodes"], cp["anc"], w.scale, cp["status"], out=cp["out"], lse=cp["lse"],
                             workspace=cp["ws"])

    def accept_call(cp):
        tvb.tree_accept(cp["target"], cp["draft"], shared["tokens"], shared["parents"], shared["n_nodes"],
                        cp["anc"], cp["depth"], w.temperature, shared["u_accept"] if sampling else None,
                        shared["u_sample"] if sampling else None, cp["status"], outputs=cp["acc"],
                        workspace=cp["aws"])

    def commit_call(cp):
        tvb.kv_commit_path(cp["k"], cp["v"], shared["page_table"], shared["prefix_len"], shared["n_nodes"],
                           cp["acc"][0], cp["acc"][1], cp["status"], outputs=cp["com"])

    def accept_commit_call(cp):
        accept_call(cp)
        commit_call(cp)

    def step_call(cp):
        mask_call(cp)
        attn_call(cp)
        accept_commit_call(cp)

    launches_per_step = tvb.launches_per_step()
    for cp in copies:                      # eager warm-up sets kernel attributes before capture
        step_call(cp)
    torch.cuda.synchronize()

    side = torch.cuda.Stream(dev)
    graphs, ac_graph = [], torch.cuda.CUDAGraph()
    acc_graph, com_graph = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        for cp in copies:
            gph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gph, stream=side):
                step_call(cp)
            graphs.append(gph)
        with torch.cuda.graph(ac_graph, stream=side):
            for cp in copies:
                accept_commit_call(cp)
        with torch.cuda.graph(acc_graph, stream=side):
            for cp in copies:
                accept_call(cp)
        with torch.cuda.graph(com_graph, stream=side):
            for cp in copies:
                commit_call(cp)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    K, Wm = args.steps, args.warmup
    for i in range(Wm):
        graphs[i % R].replay()
    barrier()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(K):
        graphs[i % R].replay()
    e1.record(stream)
    barrier()
    step_ms = e0.elapsed_time(e1) / K

    # the accept+commit pair alone, and each of the two alone, same rotation
    reps = max(3, K // R)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ac_graph.replay()
    c0.record(stream)
    for _ in range(reps):
        ac_graph.replay()
    c1.record(stream)
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    acc_graph.replay()
    x0.record(stream)
    for _ in range(reps):
        acc_graph.replay()
    x1.record(stream)
    y0, y1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    com_graph.replay()
    y0.record(stream)
    for _ in range(reps):
        com_graph.replay()
    y1.record(stream)
    torch.cuda.synchronize()
    expand = time_expand(args, W, tvb, torch, np, dev, stream, B, n_max, V, cfg)
    clk = clocks.stop()
    ac_us = c0.elapsed_time(c1) * 1000.0 / (reps * R)
    accept_us = x0.elapsed_time(x1) * 1000.0 / (reps * R)
    commit_us = y0.elapsed_time(y1) * 1000.0 / (reps * R)
    # bytes of the accept and commit rooflines: logits rows (all nodes; the accepted
    # path's nodes only, the lower bound) and the moved K/V rows of every layer
    acc_len = copies[0]["acc"][0].cpu().numpy().astype(np.int64)
    path_nodes = copies[0]["acc"][1].cpu().numpy()
    rows_factor = (2 if sampling else 1) * V * 4
    accept_bytes_all = int(np.sum(w.n_nodes)) * rows_factor
    accept_bytes_path = int(np.sum(acc_len + 1)) * rows_factor
    moved = sum(int(np.sum(path_nodes[b, 1:acc_len[b] + 1] != np.arange(1, acc_len[b] + 1)))
                for b in range(B))
    commit_bytes = moved * 2 * Hkv * D * 2 * 2 * layers  # K and V rows, read and written

    # end to end through the public binding with host buffers
    e2e = None
    if not args.no_e2e:
        host_in = dict(q=w.q_bits.view(np.int16), target=w.target_logits, parents=w.parents, n_nodes=w.n_nodes,
                       prefix_len=w.prefix_len, page_table=w.page_table, tokens=w.tokens)
        if sampling:
            host_in.update(draft=w.draft_logits, u_accept=w.u_accept, u_sample=w.u_sample)
        # every input of a step packed in one pinned buffer and one device buffer per
        # rotated copy: one host-to-device copy a step (and one copy back of the results)
        in_specs = [(k, torch.from_numpy(np.ascontiguousarray(v)).dtype, v.shape) for k, v in host_in.items()]
        _, in_bytes = packed_views(None, in_specs)
        pinned_buf = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        pinned, _ = packed_views(pinned_buf, in_specs)
        for k, v in host_in.items():
            pinned[k].copy_(torch.from_numpy(np.ascontiguousarray(v)))
        h2d_bytes = in_bytes  # the copied buffer, 256-byte padding between arrays included
        dev_bufs = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(R)]
        dev_ins = [packed_views(b, in_specs)[0] for b in dev_bufs]
        res_host_buf = torch.empty(res_bytes, dtype=torch.uint8).pin_memory()
        res_host_v, _ = packed_views(res_host_buf, res_specs)
        res_names = ["accept_len", "path_nodes", "out_tokens", "new_len", "slots"]
        res_host = [res_host_v[n] for n in res_names]
        d2h = res_bytes

        def h2d(k):
            dev_bufs[k % R].copy_(pinned_buf, non_blocking=True)

        def compute(k):
            cpk = copies[k % R]
            dev_in = dev_ins[k % R]
            anc, depth, st = tvb.tree_build_mask(dev_in["parents"], dev_in["n_nodes"], anc_mask=cpk["anc"],
                                                 depth=cpk["depth"], status=cpk["status"])
            tvb.tree_verify_attn(dev_in["q"].view(torch.bfloat16), cpk["k"][0], cpk["v"][0], dev_in["page_table"],
                                 dev_in["prefix_len"], dev_in["n_nodes"], anc, w.scale, st, out=cpk["out"],
                                 lse=cpk["lse"], workspace=cpk["ws"])
            acc = tvb.tree_accept(dev_in["target"], dev_in.get("draft"), dev_in["tokens"], dev_in["parents"],
                                  dev_in["n_nodes"], anc, depth, w.temperature, dev_in.get("u_accept"),
                                  dev_in.get("u_sample"), st, outputs=cpk["acc"], workspace=cpk["aws"])
            com = tvb.kv_commit_path(cpk["k"], cpk["v"], dev_in["page_table"], dev_in["prefix_len"],
                                     dev_in["n_nodes"], acc[0], acc[1], st, outputs=cpk["com"])
            res_host_buf.copy_(cpk["res"], non_blocking=True)

        def e2e_step(k):
            h2d(k)
            compute(k)

        K2 = min(K, 500)
        for k in range(min(Wm, 5)):
            e2e_step(k)
        barrier()
        # (a) one python call per library function and per copy, every step
        t_start = time.perf_counter()
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(stream)
        for k in range(K2):
            e2e_step(k)
        x1.record(stream)
        barrier()
        wall = time.perf_counter() - t_start
        eager_ms = max(x0.elapsed_time(x1), wall * 1000.0) / K2
        # (b) the same step captured once per rotated copy as a CUDA graph (host->device
        # copies from pinned memory, the four calls, device->host copies of the results)
        # and replayed: how a serving loop drives the library
        e2e_graphs = []
        with torch.cuda.stream(side):
            for k in range(R):
                gph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gph, stream=side):
                    e2e_step(k)
                e2e_graphs.append(gph)
        torch.cuda.synchronize()
        for k in range(min(Wm, 5)):
            e2e_graphs[k % R].replay()
        barrier()
        for t in res_host:
            t.fill_(-7)
        t_start = time.perf_counter()
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(stream)
        for k in range(K2):
            e2e_graphs[k % R].replay()
        x1.record(stream)
        barrier()
        wall = time.perf_counter() - t_start
        graph_ms = max(x0.elapsed_time(x1), wall * 1000.0) / K2
        last = copies[(K2 - 1) % R]
        landed = all(torch.equal(h, d.cpu()) for h, d in zip(
            res_host, [last["acc"][0], last["acc"][1], last["acc"][2], last["com"][1], last["com"][0]]))
        # (c) pipelined: one CUDA graph per step holds the host->device copy of the next
        # step's inputs on a copy stream (forked from and joined back into the graph)
        # beside this step's compute; each rotated copy has its own input buffers, so
        # the copy never writes what the compute reads, and consecutive graphs run in
        # order, so step k+1 reads what graph k copied. The host issues one replay a step.
        copy_stream = torch.cuda.Stream(dev)
        pipe_graphs = []
        with torch.cuda.stream(side):
            for k in range(R):
                gph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gph, stream=side):
                    copy_stream.wait_stream(side)      # fork
                    with torch.cuda.stream(copy_stream):
                        h2d(k + 1)
                    compute(k)
                    side.wait_stream(copy_stream)      # join
                pipe_graphs.append(gph)
        torch.cuda.synchronize()
        h2d(0)
        torch.cuda.synchronize()

        def pipelined(n):
            for i in range(n):
                pipe_graphs[i % R].replay()
        pipelined(min(Wm, 5))
        barrier()
        for t in res_host:
            t.fill_(-7)
        t_start = time.perf_counter()
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(stream)
        pipelined(K2)
        x1.record(stream)
        barrier()
        wall = time.perf_counter() - t_start
        pipe_ms = max(x0.elapsed_time(x1), wall * 1000.0) / K2
        landed = landed and all(torch.equal(h, d.cpu()) for h, d in zip(
            res_host, [last["acc"][0], last["acc"][1], last["acc"][2], last["com"][1], last["com"][0]]))
        nodes_b = float(np.sum(w.n_nodes))
        e2e = {"value": nodes_b / (pipe_ms / 1000.0), "unit": "nodes/s",
               "h2d_bytes_per_step": int(h2d_bytes), "d2h_bytes_per_step": int(d2h), "ms_per_step": pipe_ms,
               "steps": K2, "results_landed_on_host": bool(landed),
               "note": "per step: queries, tree, logits and uniforms copied from pinned host memory, mask + "
                       "attention + accept + commit through the library, results copied back to pinned host "
                       "memory; one CUDA graph per step, holding the copy of the next step's inputs on a second "
                       "stream beside this step's compute; KV cache resident in HBM; wall clock and events, the "
                       "larger",
               "serial_graph": {"value": nodes_b / (graph_ms / 1000.0), "ms_per_step": graph_ms,
                                "note": "copy, compute and copy back in one CUDA graph per step, no overlap"},
               "eager": {"value": nodes_b / (eager_ms / 1000.0), "ms_per_step": eager_ms,
                         "note": "the same step as one python binding call per function and per copy"}}

    # each Llama-shaped workload's attention on its own, this config's first (the
    # headline roofline), each over >= --leg-seconds with its SM clocks sampled
    del copies, graphs, ac_graph, acc_graph, com_graph
    torch.cuda.empty_cache()
    leg_names = [cfg.name] + [n for n in ("llama3_70b", "long", "serving", "llama2_7b") if n != cfg.name]
    legs = attn_legs(W, tvb, dev, local_rank, leg_names, min_seconds=args.leg_seconds,
                     q4_seconds=args.leg_seconds / 2)
    attn_us = legs[cfg.name]["us"]

    nodes = float(np.sum(w.n_nodes))
    e2e_in = [e2e["ms_per_step"], e2e["eager"]["ms_per_step"], e2e["serial_graph"]["ms_per_step"]] \
        if e2e is not None else []
    (step_ms, attn_us, ac_us, accept_us, commit_us, expand_us, *e2e_out), (nodes_total,) = reduce_over_ranks(
        [step_ms, attn_us, ac_us, accept_us, commit_us, expand["us_per_tree"]] + e2e_in, [nodes], dev)
    expand["us_per_tree"] = expand_us
    if e2e is not None:
        e2e["ms_per_step"] = e2e_out[0]
        e2e["value"] = nodes_total / (e2e["ms_per_step"] / 1000.0)
        e2e["eager"]["ms_per_step"] = e2e_out[1]
        e2e["eager"]["value"] = nodes_total / (e2e_out[1] / 1000.0)
        e2e["serial_graph"]["ms_per_step"] = e2e_out[2]
        e2e["serial_graph"]["value"] = nodes_total / (e2e_out[2] / 1000.0)

    hbm, tf_burst, peak_src = load_peaks()
    abytes, aflops = w.attn_bytes(), w.attn_flops()
    attn_s = attn_us * 1e-6
    roof = attn_roofline(abytes, aflops, attn_us, hbm, tf_burst, load_traffic(cfg.name))
    roof.update(peak_source=f"{peak_src} (MEASURED_PEAKS.json, burst)", kernel="tv_tree_verify_attn",
                timed=f"{legs[cfg.name]['launches']} launches over {legs[cfg.name]['timed_s']:.2f} s, "
                      f"{legs[cfg.name]['rotated_copies']} rotated cache copies (> 3x L2)",
                clocks=legs[cfg.name]["clocks"],
                algorithmic={"bytes": abytes, "flops": aflops, "exps": aflops // (4 * D), "out_bytes": w.out_bytes()})
    acc_mean = float(np.mean(acc_len))
    acceptance = {"mode": f"sampling T={w.temperature}" if sampling else "greedy",
                  "sibling_rule": ("fixed draft (siblings drawn i.i.d. from q, as this workload draws them)"
                                   if sampling else "argmax"),
                  "mean_accept_len": acc_mean, "tokens_per_step": acc_mean + 1.0,
                  "accept_len_per_request": acc_len.tolist(),
                  "note": "synthetic logits (Gaussian, rho-correlated draft): acceptance is a property of these "
                          "inputs, not of a trained drafter"}

    line = {
        "metric": METRIC,
        "value": nodes_total / (step_ms / 1000.0),
        "unit": "nodes/s",
        "n_gpus": world,
        "steps": K,
        "warmup": Wm,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded numpy PCG64; random bf16 KV/Q ~ N(0,1), Gaussian fp32 logits)",
        "config": dict(workload_config(cfg, world),
                       l2=f"{R} rotated input copies ({R * per_copy / 1e6:.0f} MB read per rotation) > 3x L2",
                       step="mask + attention + accept + commit, one CUDA graph replay"),
        "attn_us": attn_us,
        "attn_tbps": abytes / attn_s / 1e12,
        "attn_roofline_frac": roof["frac"],
        "attn_nodes_per_s": nodes_total / attn_s,
        "attn_legs": legs,
        "acceptance": acceptance,
        "accept_commit_us": ac_us,
        "accept": {"us": accept_us, "mode": "sampling" if sampling else "greedy",
                   "bytes_all_rows": accept_bytes_all, "bytes_path_rows": accept_bytes_path,
                   "hbm_us_all_rows": accept_bytes_all / (hbm * 1e3),
                   "hbm_us_path_rows": accept_bytes_path / (hbm * 1e3)},
        "commit": {"us": commit_us, "layers": layers, "moved_rows_per_layer_head": moved,
                   "bytes": commit_bytes, "bytes_one_layer": commit_bytes // max(layers, 1),
                   "hbm_us": commit_bytes / (hbm * 1e3)},
        "nodes_per_s_attn_accept_commit": nodes_total / ((attn_us + accept_us + commit_us) * 1e-6),
        "attn_q4": dict(legs[cfg.name]["q4"], cache="the same K/V encoded by tv_kv_quantize_q4"),
        "expand": dict(expand, us_per_level=expand_us / expand["levels"],
                       hbm_us=expand["bytes"] / (hbm * 1e3), hbm_frac=expand["bytes"] / (hbm * 1e3) / expand_us),
        "roofline": roof,
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline:
        try:
            line["cpu_baseline"] = cpu_baseline_obj(oracle_leg_subprocess(args.config))
        except Exception as ex:  # report it, keep the GPU line
            line["cpu_baseline"] = {"value": None, "error": str(ex)[:300]}
        try:
            ref = oracle_accept_subprocess(args.config)
            nb = np.asarray(ref["near_boundary"], dtype=bool)
            line["acceptance"].update(
                near_boundary_requests=int(nb.sum()),
                oracle_accept_len=ref["accept_len"],
                matches_oracle=bool(np.array_equal(acc_len[~nb], np.asarray(ref["accept_len"])[~nb])),
                oracle_note="the fp64 oracle's acceptance on the same inputs; a request with a decision within "
                            "1e-6 of its threshold is near-boundary and excused")
        except Exception as ex:
            line["acceptance"]["oracle_error"] = str(ex)[:300]
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_reference(args, world, rank):
    """The oracle as it stands, on the host cores (the attention rows spread
    over every core, the rest single-thread), on bounded samples of the same
    workload."""
    if rank != 0:
        return
    import numpy as np
    from eagle_speculative_decoding_attn_gb300 import workloads as W
    steps = max(1, min(args.steps, 3))
    warm = 1 if args.warmup > 0 else 0
    for _ in range(warm):
        oracle_leg_subprocess(args.config)
    res, times = None, []
    for _ in range(steps):
        res = oracle_leg_subprocess(args.config)
        times.append(res["seconds_per_step_all_cores"])
    sps = float(np.mean(times))
    value = res["nodes"] / sps
    print(json.dumps({"impl": "reference", "metric": METRIC, "value": value, "unit": "nodes/s", "n_gpus": world,
                      "steps": steps, "warmup": warm, "ms_per_step": sps * 1000.0, "higher_is_better": True,
                      "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                      "config": workload_config(W.CONFIG_BY_NAME[args.config], world),
                      "cpu_baseline": {"value": value, "unit": "nodes/s", "cores": res["cores"], "kind": "oracle",
                                       "sample": res["desc"] + "; attention rows spread over the cores"},
                      "e2e": {"value": value, "unit": "nodes/s", "h2d_bytes_per_step": 0,
                              "d2h_bytes_per_step": 0}}))


if __name__ == "__main__":
    main()
