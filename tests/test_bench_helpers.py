"""Host-side helpers of bench.py: packed host/device buffers (one copy each way
per step) and the workload config both arms print."""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from eagle_speculative_decoding_attn_gb300 import workloads as W  # noqa: E402


def test_packed_views_are_aligned_disjoint_and_round_trip():
    specs = [("a", torch.int32, (3,)), ("b", torch.int64, (5, 7)), ("c", torch.float32, (2, 3, 4)),
             ("d", torch.int16, (9,)), ("e", torch.int64, (1,))]
    _, total = bench.packed_views(None, specs)
    buf = torch.zeros(total, dtype=torch.uint8)
    views, total2 = bench.packed_views(buf, specs)
    assert total2 == total and total % 256 == 0
    spans = []
    for name, dtype, shape in specs:
        v = views[name]
        assert v.dtype == dtype and tuple(v.shape) == shape and v.is_contiguous()
        off = v.data_ptr() - buf.data_ptr()
        assert off % 256 == 0
        spans.append((off, off + v.numel() * v.element_size()))
    spans.sort()
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))  # no overlap
    rng = np.random.default_rng(0)
    for name, dtype, shape in specs:
        x = torch.from_numpy(rng.integers(-100, 100, size=shape)).to(dtype)
        views[name].copy_(x)
    again, _ = bench.packed_views(buf.clone(), specs)       # a copy of the buffer carries every array
    for name, _, _ in specs:
        assert torch.equal(again[name], views[name])


def test_both_arms_name_the_workload_alike():
    for cfg in W.CONFIGS:
        c1 = bench.workload_config(cfg, 1)
        assert c1["workload"].startswith(cfg.name + ":") and c1["global_batch"] == cfg.B
        assert bench.workload_config(cfg, 4)["global_batch"] == 4 * cfg.B
