"""A bounded wait that runs out on the GPU: the self-test kernel waits on an
mbarrier nothing completes (the same wait routine as every kernel), gives up
after its limit, reports TV_DEV_TIMEOUT, and the context stays usable."""
import time

import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
from eagle_speculative_decoding_attn_gb300 import workloads as W
from gpu_helpers import DevWorkload, require_gpu

pytestmark = pytest.mark.gpu


def test_wait_limit_expires_and_reports_timeout():
    dev = require_gpu()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    t0 = time.perf_counter()
    tvb.selftest_wait_timeout(status)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status.item()) == oracle.STATUS_TIMEOUT
    assert 0.9 < dt < 30.0
    # the context still runs work afterwards
    w = W.make_workload("tiny", with_logits=False)
    anc, depth, st = DevWorkload(w, dev, logits=False).mask()
    ref_anc, _, ref_st = oracle.tree_build_mask(w.parents, w.n_nodes)
    assert np.array_equal(anc.cpu().numpy().view(np.uint64), ref_anc) and np.array_equal(st.cpu().numpy(), ref_st)
