"""Pins of the oracle's 4-bit KV decoding and quantised attention (no GPU).

Source: troisinh.com "EAGLE - Draft head ..." (EAGLE pairs with an INT4 KV
cache; further reading: KV-cache quantisation to INT4/INT3).  Pinned by a
hand-worked row (tests/golden/q4_example.txt), torch's own float32 -> bfloat16
cast, the code-0 / code-15 ends and monotonicity, and an exactly representable
cache (scale 1, zero -8) on which the quantised attention must equal the bf16
attention of the integer values written out independently.
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_attn_gb300 import workloads as W
from golden_io import read_fixture


def test_hand_worked_row():
    fx = read_fixture("q4_example.txt")
    prm = [float(x) for x in fx["params"]]
    codes = np.zeros((1, 32), np.uint8)
    for kv in fx["bytes_set"]:
        j, v = kv.split("=")
        codes[0, int(j)] = int(v, 16)
    params = np.array([prm], np.float16)
    bits = oracle.dequantize_q4(codes, params)
    dims = [int(d) for d in fx["dims"]]
    assert [int(bits[0, d]) for d in dims] == [int(b, 16) for b in fx["bits"]]


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    ties = (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32).astype(np.float64)
    ties = np.concatenate([ties, (np.uint32(0x3F810000) | np.uint32(0x8000)).reshape(1).view(np.float32)])
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-6, 6, 20000),
                        [0.0, -0.0, 1.0, 3.140625, 65504.0, 1e-30], ties, -ties])
    ours = oracle.f64_to_bf16_bits_via_f32(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_code_ends_and_monotone():
    rng = np.random.default_rng(2)
    D = 128
    s = rng.uniform(0.1, 0.4, size=(50, 4)).astype(np.float16)
    z = rng.normal(0, 1, size=(50, 4)).astype(np.float16)
    params = np.empty((50, 8), np.float16)
    params[:, 0::2], params[:, 1::2] = s, z
    vals = []
    for c in range(16):
        codes = np.full((50, D // 2), c | (c << 4), np.uint8)
        vals.append(oracle.bf16_to_f64(oracle.dequantize_q4(codes, params)))
    g = np.repeat(np.arange(4), 32)
    np.testing.assert_array_equal(vals[0], oracle.bf16_to_f64(oracle.f64_to_bf16_bits_via_f32(
        z.astype(np.float64)[:, g])))
    np.testing.assert_array_equal(vals[15], oracle.bf16_to_f64(oracle.f64_to_bf16_bits_via_f32(
        15.0 * s.astype(np.float64)[:, g] + z.astype(np.float64)[:, g])))
    for c in range(15):
        assert np.all(vals[c + 1] >= vals[c])


def test_exact_cache_equals_bf16_attention():
    """K with scale 1, zero -8 and V with scale 2, zero -15 decode to small
    integers (exact in bf16): the quantised attention equals the bf16
    attention over those integers."""
    w = W.make_custom(B=2, Hq=4, Hkv=2, D=128, prefix_len=[37, 5], parents_list=[W.chain_tree(5), [-1, 0, 0, 1]],
                      seed=4)
    rng = np.random.default_rng(5)
    shape = w.k_bits.shape
    kc = rng.integers(0, 256, size=shape[:-1] + (64,), dtype=np.uint8)
    vc = rng.integers(0, 256, size=shape[:-1] + (64,), dtype=np.uint8)
    kp = np.zeros(shape[:-1] + (8,), np.float16)
    kp[..., 0::2], kp[..., 1::2] = 1.0, -8.0
    vp = np.zeros(shape[:-1] + (8,), np.float16)
    vp[..., 0::2], vp[..., 1::2] = 2.0, -15.0      # V decodes to 2c - 15

    def ints(codes, a, b):
        out = np.empty(codes.shape[:-1] + (128,), np.float32)
        out[..., 0::2] = a * (codes & 15).astype(np.float32) + b
        out[..., 1::2] = a * (codes >> 4).astype(np.float32) + b
        return torch.from_numpy(out).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)

    o1, l1, s1 = oracle.tree_verify_attn_q4(w.q_bits, kc, kp, vc, vp, w.page_table, w.prefix_len,
                                            w.n_nodes, w.parents, w.scale)
    o2, l2, s2 = oracle.tree_verify_attn(w.q_bits, ints(kc, 1, -8), ints(vc, 2, -15), w.page_table, w.prefix_len,
                                         w.n_nodes, w.parents, w.scale)
    assert np.array_equal(s1, s2)
    np.testing.assert_array_equal(np.nan_to_num(o1, nan=7.0), np.nan_to_num(o2, nan=7.0))
    np.testing.assert_array_equal(np.nan_to_num(l1, nan=7.0), np.nan_to_num(l2, nan=7.0))


def test_generated_cache_spread():
    rng = np.random.default_rng(6)
    codes, params = W.make_q4_cache(rng, 20, 2, 128)
    v = oracle.bf16_to_f64(oracle.dequantize_q4(codes, params))
    assert abs(v.mean()) < 0.05 and 0.7 < v.std() < 1.3


# --------------------------------------------------------------------------
# the encoder
# --------------------------------------------------------------------------
def _bits(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_quantize_hand_worked_group():
    # group 0: values 0.0, 1.5, 3.0 ... (0.25 steps): min 0, max 7.5 -> scale 0.5, codes x / 0.5
    D = 64
    x = np.zeros(D, np.float32)
    x[:32] = np.arange(32) * 0.25 % 7.75          # 0 .. 7.5 in quarter steps
    x[32:] = -1.0                                 # group 1 constant: scale 0, codes 0
    codes, params = oracle.quantize_q4(_bits(x))
    assert params.astype(np.float32).tolist() == [0.5, 0.0, 0.0, -1.0]
    c = np.empty(D, np.int64)
    c[0::2], c[1::2] = codes & 15, codes >> 4
    expect = np.rint(x[:32] / 0.5).astype(np.int64)     # ties to even: 0.25 / 0.5 = 0.5 -> 0, 0.75 -> 2
    assert c[:32].tolist() == expect.tolist()
    assert c[32:].tolist() == [0] * 32
    assert oracle.bf16_to_f64(oracle.dequantize_q4(codes, params))[32:].tolist() == [-1.0] * 32


def test_quantize_round_trip_error_bound():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((300, 128)).astype(np.float32) * rng.uniform(0.1, 5, size=(300, 1)).astype(np.float32)
    xb = _bits(x)
    codes, params = oracle.quantize_q4(xb)
    back = oracle.bf16_to_f64(oracle.dequantize_q4(codes, params))
    xv = oracle.bf16_to_f64(xb)
    s = np.repeat(params[:, 0::2].astype(np.float64), 32, axis=1)
    z = np.repeat(params[:, 1::2].astype(np.float64), 32, axis=1)
    # half a step, plus the fp16 rounding of zero and scale (at most 15 steps of it), plus bf16 output rounding
    bound = 0.5 * s + np.abs(xv.reshape(300, 4, 32).min(-1).repeat(32, 1) - z) + 15 * s * 2.0 ** -11 \
        + np.abs(back) * 2.0 ** -8
    assert np.all(np.abs(back - xv) <= bound + 1e-12)
    # codes reach both ends of every non-constant group
    q = np.empty((300, 128), np.int64)
    q[:, 0::2], q[:, 1::2] = codes & 15, codes >> 4
    assert (q.reshape(300, 4, 32).min(-1) == 0).all()
    assert (q.reshape(300, 4, 32).max(-1) >= 14).all()


def test_quantize_codes_match_float32_definition():
    """Each code is rint((x - zero) * fp32(1 / scale)) in float32, written out
    with Python's own float rounding of every step (struct pack to float32)."""
    import struct
    f32 = lambda v: struct.unpack("f", struct.pack("f", v))[0]
    rng = np.random.default_rng(8)
    x = rng.standard_normal((20, 64)).astype(np.float32)
    codes, params = oracle.quantize_q4(_bits(x))
    xv = oracle.bf16_to_f64(_bits(x))
    for r in range(20):
        for d in range(64):
            grp = d // 32
            s, z = float(params[r, 2 * grp]), float(params[r, 2 * grp + 1])
            c = round(f32(f32(xv[r, d] - z) * f32(1.0 / s)))   # Python round: half to even
            c = min(15, max(0, c))
            got = (codes[r, d // 2] >> (4 * (d % 2))) & 15
            assert got == c


def _fp16_round_exact(fr):
    """The float16 nearest to the rational fr (ties to even mantissa), found by
    exact comparison with the neighbours of a first guess."""
    from fractions import Fraction
    g = np.float16(float(fr))
    cands = {g, np.nextafter(g, np.float16(np.inf)), np.nextafter(g, np.float16(-np.inf))}
    best = None
    for c in cands:
        if not np.isfinite(c):
            continue
        d = abs(Fraction(float(c)) - fr)
        even = (int(np.array(c, np.float16).view(np.uint16)) & 1) == 0
        key = (d, not even)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_quantize_against_exact_rational_rounding():
    """The encoder's integer decisions against exact arithmetic (Python
    fractions), independent of its float32 steps.

    Parameters: zero is the float16 nearest to the group minimum and scale the
    float16 nearest to (max - min) / 15, both rounded exactly here.  Codes: the
    nearest integer (ties to even) to the exact rational (x - zero) / scale,
    clamped to [0, 15], for the stored (scale, zero).  The float32 form rounds
    x - zero, 1 / scale and their product once each (relative error at most
    3 * 2^-24 of a quotient <= 15.5), so a code may differ from the exact one
    only where the exact quotient lies within 16 * 3 * 2^-24 of a half-integer;
    every differing code is checked to be such a case and the count is bounded."""
    from fractions import Fraction
    rng = np.random.default_rng(21)
    rows = [rng.standard_normal((600, 128)).astype(np.float32),                       # the workloads' N(0, 1)
            (rng.standard_normal((200, 128)) * rng.uniform(1e-3, 50, (200, 1))).astype(np.float32),
            rng.integers(-8, 8, (50, 128)).astype(np.float32) * 0.5]                 # exact steps, many ties
    x = np.concatenate(rows)
    xb = _bits(x)
    codes, params = oracle.quantize_q4(xb)
    xv = oracle.bf16_to_f64(xb)
    n_rows, D = xv.shape
    q = np.empty((n_rows, D), np.int64)
    q[:, 0::2], q[:, 1::2] = codes & 15, codes >> 4
    slack = Fraction(16 * 3, 2 ** 24)
    n_codes = n_diff = n_param_diff = 0
    for r in range(n_rows):
        for grp in range(D // 32):
            vals = [Fraction(float(v)) for v in xv[r, 32 * grp: 32 * grp + 32]]
            mn, mx = min(vals), max(vals)
            s_ex = _fp16_round_exact((mx - mn) / 15)
            z_ex = _fp16_round_exact(mn)
            s_got, z_got = params[r, 2 * grp], params[r, 2 * grp + 1]
            assert z_got == z_ex, (r, grp)
            if s_got != s_ex:
                # float32 then float16 (double rounding) may differ from one exact rounding
                # only next to a float16 tie
                n_param_diff += 1
                assert abs(float(s_got) - float(s_ex)) <= float(np.spacing(np.float16(s_ex))), (r, grp)
            s, z = Fraction(float(s_got)), Fraction(float(z_got))
            for d in range(32):
                n_codes += 1
                got = int(q[r, 32 * grp + d])
                if s == 0:
                    assert got == 0
                    continue
                t = (vals[d] - z) / s
                exact = min(15, max(0, round(t)))          # round() of a Fraction: ties to even
                if got != exact:
                    n_diff += 1
                    half = Fraction(2 * min(got, exact) + 1, 2)
                    assert abs(got - exact) == 1 and abs(t - half) <= slack, (r, grp, d, float(t))
    assert n_codes == n_rows * D
    assert n_diff <= n_codes // 10000, n_diff
    assert n_param_diff <= (n_rows * D // 32) // 1000, n_param_diff
    print(f"exact-rounding pin: {n_diff} of {n_codes} codes and {n_param_diff} scales differ (all at ties)")
