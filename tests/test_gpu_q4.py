"""GPU parity of tv_kv_quantize_q4 against the oracle's encoder: codes and
parameters bit-exact (both take the integer decisions in float32 IEEE steps
with fp16 parameters)."""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
from eagle_speculative_decoding_attn_gb300 import workloads as W
from gpu_helpers import bf16_dev, require_gpu

pytestmark = pytest.mark.gpu


def _check(bits, dev):
    x = bf16_dev(bits, dev)
    codes, params = tvb.kv_quantize_q4(x)
    torch.cuda.synchronize()
    rc, rp = oracle.quantize_q4(bits)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(params.cpu().numpy().view(np.uint16), rp.view(np.uint16))


@pytest.mark.parametrize("D,rows,seed", [(32, 1, 0), (64, 333, 1), (128, 5000, 2), (256, 77, 3)])
def test_random_rows(D, rows, seed):
    dev = require_gpu()
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, D)) * rng.uniform(1e-3, 50, size=(rows, 1))).astype(np.float32)
    _check(W.to_bf16_bits(x), dev)


def test_constant_groups_ties_and_extremes():
    dev = require_gpu()
    rng = np.random.default_rng(4)
    rows = []
    rows.append(np.full(128, 3.0))                                   # constant: scale 0
    rows.append(np.repeat([0.0, 1.0, -2.5, 7.0], 32))                # constant per group
    rows.append(np.tile(np.arange(32) * 0.25, 4))                    # quarter steps: ties at .5
    rows.append(np.tile(np.linspace(-1, 1, 32), 4) * 60000.0)        # near the fp16 range
    rows.append(np.tile(np.linspace(0, 1, 32), 4) * 1e-6)            # tiny: fp16 subnormal scales
    rows.append(rng.integers(-8, 8, size=128).astype(np.float64))    # small integers
    x = np.stack(rows).astype(np.float32)
    _check(W.to_bf16_bits(x), dev)


def test_paged_cache_llama2_7b_shape():
    """A whole layer of the 7B-shaped paged cache, [pages, Hkv, 16, 128]."""
    dev = require_gpu()
    w = W.make_workload("llama2_7b", with_logits=False)
    _check(w.k_bits, dev)


def test_round_trip_through_decoder():
    dev = require_gpu()
    rng = np.random.default_rng(5)
    bits = W.to_bf16_bits(rng.standard_normal((64, 128)).astype(np.float32))
    codes, params = tvb.kv_quantize_q4(bf16_dev(bits, dev))
    back = oracle.bf16_to_f64(oracle.dequantize_q4(codes.cpu().numpy(), params.cpu().numpy()))
    xv = oracle.bf16_to_f64(bits)
    s = np.repeat(params.cpu().numpy()[:, 0::2].astype(np.float64), 32, axis=1)
    assert np.all(np.abs(back - xv) <= 0.6 * s + np.abs(xv) * 2.0 ** -7 + 1e-3 * s)
