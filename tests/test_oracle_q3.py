"""Pins of the oracle's 3-bit KV format, encoder and quantised attention (no GPU).

Source: troisinh.com "EAGLE - Draft head ..." (further reading: KV-cache
quantisation to INT4/INT3).  Pinned by a hand-worked row
(tests/golden/q3_example.txt), a bit-by-bit restatement of the layout, the
code-0 / code-7 ends and monotonicity, an exactly representable cache on which
the quantised attention must equal the bf16 attention of the integers written
out independently, and the encoder against float32 arithmetic written out with
Python's own rounding and against exact rational rounding.
"""
from fractions import Fraction

import numpy as np
import torch

import oracle
from golden_io import read_fixture
from test_oracle_q4 import _fp16_round_exact
from eagle_speculative_decoding_attn_gb300 import workloads as W


def _bits(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_hand_worked_row():
    fx = read_fixture("q3_example.txt")
    codes = np.zeros((1, 24), np.uint8)
    for kv in fx["bytes_set"]:
        j, v = kv.split("=")
        codes[0, int(j)] = int(v, 16)
    params = np.array([[float(x) for x in fx["params"]]], np.float16)
    bits = oracle.dequantize_q3(codes, params)
    dims = [int(d) for d in fx["dims"]]
    assert [int(bits[0, d]) for d in dims] == [int(b, 16) for b in fx["bits"]]


def test_layout_bit_by_bit():
    """The packing against the layout restated one bit at a time."""
    rng = np.random.default_rng(11)
    for D in (32, 64, 128):
        c = rng.integers(0, 8, size=(7, D))
        packed = oracle.q3_pack(c)
        assert packed.shape == (7, 3 * D // 8)
        for r in range(7):
            want = [0] * (3 * D // 8)
            for d in range(D):
                code = int(c[r, d])
                byte, pos = d // 4, 2 * (d % 4)              # low two bits
                want[byte] |= (code & 3) << pos
                byte, pos = D // 4 + d // 8, d % 8           # third bit
                want[byte] |= ((code >> 2) & 1) << pos
            assert packed[r].tolist() == want
        assert np.array_equal(oracle.q3_code_values(packed, D), c)


def test_code_ends_and_monotone():
    rng = np.random.default_rng(2)
    D = 128
    s = rng.uniform(0.1, 0.4, size=(50, 4)).astype(np.float16)
    z = rng.normal(0, 1, size=(50, 4)).astype(np.float16)
    params = np.empty((50, 8), np.float16)
    params[:, 0::2], params[:, 1::2] = s, z
    g = np.repeat(np.arange(4), 32)
    vals = []
    for c in range(8):
        codes = oracle.q3_pack(np.full((50, D), c))
        vals.append(oracle.bf16_to_f64(oracle.dequantize_q3(codes, params)))
    np.testing.assert_array_equal(vals[0], oracle.bf16_to_f64(oracle.f64_to_bf16_bits_via_f32(
        z.astype(np.float64)[:, g])))
    np.testing.assert_array_equal(vals[7], oracle.bf16_to_f64(oracle.f64_to_bf16_bits_via_f32(
        7.0 * s.astype(np.float64)[:, g] + z.astype(np.float64)[:, g])))
    for c in range(7):
        assert np.all(vals[c + 1] >= vals[c])


def test_exact_cache_equals_bf16_attention():
    """K with scale 1, zero -4 and V with scale 2, zero -7 decode to small
    integers (exact in bf16): the quantised attention equals the bf16
    attention over those integers."""
    w = W.make_custom(B=2, Hq=4, Hkv=2, D=128, prefix_len=[37, 5], parents_list=[W.chain_tree(5), [-1, 0, 0, 1]],
                      seed=4)
    rng = np.random.default_rng(5)
    shape = w.k_bits.shape
    kc = rng.integers(0, 8, size=shape)
    vc = rng.integers(0, 8, size=shape)
    kp = np.zeros(shape[:-1] + (8,), np.float16)
    kp[..., 0::2], kp[..., 1::2] = 1.0, -4.0
    vp = np.zeros(shape[:-1] + (8,), np.float16)
    vp[..., 0::2], vp[..., 1::2] = 2.0, -7.0      # V decodes to 2c - 7
    o1, l1, s1 = oracle.tree_verify_attn_q3(w.q_bits, oracle.q3_pack(kc), kp, oracle.q3_pack(vc), vp,
                                            w.page_table, w.prefix_len, w.n_nodes, w.parents, w.scale)
    o2, l2, s2 = oracle.tree_verify_attn(w.q_bits, _bits(kc - 4.0), _bits(2.0 * vc - 7.0), w.page_table,
                                         w.prefix_len, w.n_nodes, w.parents, w.scale)
    assert np.array_equal(s1, s2)
    np.testing.assert_array_equal(np.nan_to_num(o1, nan=7.0), np.nan_to_num(o2, nan=7.0))
    np.testing.assert_array_equal(np.nan_to_num(l1, nan=7.0), np.nan_to_num(l2, nan=7.0))


def test_quantize_hand_worked_group():
    # group 0: 0.0, 0.25, ..., steps of 0.25 mod 3.75: min 0, max 3.5 -> scale 0.5, codes rint(x / 0.5)
    D = 64
    x = np.zeros(D, np.float32)
    x[:32] = np.arange(32) * 0.25 % 3.75
    x[32:] = 2.0                                   # group 1 constant: scale 0, codes 0
    codes, params = oracle.quantize_q3(_bits(x))
    assert params.astype(np.float32).tolist() == [0.5, 0.0, 0.0, 2.0]
    c = oracle.q3_code_values(codes, D)
    expect = np.rint(x[:32] / 0.5).astype(np.int64)    # ties to even: 0.25 / 0.5 = 0.5 -> 0, 0.75 -> 2
    assert c[:32].tolist() == expect.tolist()
    assert c[32:].tolist() == [0] * 32
    assert oracle.bf16_to_f64(oracle.dequantize_q3(codes, params))[32:].tolist() == [2.0] * 32


def test_quantize_round_trip_error_bound():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((300, 128)).astype(np.float32) * rng.uniform(0.1, 5, size=(300, 1)).astype(np.float32)
    xb = _bits(x)
    codes, params = oracle.quantize_q3(xb)
    back = oracle.bf16_to_f64(oracle.dequantize_q3(codes, params))
    xv = oracle.bf16_to_f64(xb)
    s = np.repeat(params[:, 0::2].astype(np.float64), 32, axis=1)
    z = np.repeat(params[:, 1::2].astype(np.float64), 32, axis=1)
    # half a step, plus the fp16 rounding of zero and scale (at most 7 steps of it), plus bf16 output rounding
    bound = 0.5 * s + np.abs(xv.reshape(300, 4, 32).min(-1).repeat(32, 1) - z) + 7 * s * 2.0 ** -11 \
        + np.abs(back) * 2.0 ** -8
    assert np.all(np.abs(back - xv) <= bound + 1e-12)
    q = oracle.q3_code_values(codes, 128)
    assert (q.reshape(300, 4, 32).min(-1) == 0).all()
    assert (q.reshape(300, 4, 32).max(-1) >= 6).all()


def test_quantize_codes_match_float32_definition():
    """Each code is rint((x - zero) * fp32(1 / scale)) in float32, written out
    with Python's own float rounding of every step (struct pack to float32)."""
    import struct
    f32 = lambda v: struct.unpack("f", struct.pack("f", v))[0]
    rng = np.random.default_rng(8)
    x = rng.standard_normal((20, 64)).astype(np.float32)
    codes, params = oracle.quantize_q3(_bits(x))
    xv = oracle.bf16_to_f64(_bits(x))
    got_all = oracle.q3_code_values(codes, 64)
    for r in range(20):
        for d in range(64):
            grp = d // 32
            s, z = float(params[r, 2 * grp]), float(params[r, 2 * grp + 1])
            c = round(f32(f32(xv[r, d] - z) * f32(1.0 / s)))   # Python round: half to even
            assert got_all[r, d] == min(7, max(0, c))


def test_quantize_against_exact_rational_rounding():
    """The encoder's integer decisions against exact arithmetic (Python
    fractions), independent of its float32 steps: zero and scale are the
    float16 values nearest to the group minimum and (max - min) / 7, each code
    the nearest integer (ties to even) to the exact (x - zero) / scale for the
    stored parameters, clamped to [0, 7].  The float32 form rounds three times
    (relative error at most 3 * 2^-24 of a quotient <= 7.5), so a code may
    differ only where the exact quotient lies within 8 * 3 * 2^-24 of a
    half-integer; each differing code is checked to be such a case."""
    rng = np.random.default_rng(21)
    rows = [rng.standard_normal((600, 128)).astype(np.float32),
            (rng.standard_normal((200, 128)) * rng.uniform(1e-3, 50, (200, 1))).astype(np.float32),
            rng.integers(-4, 4, (50, 128)).astype(np.float32) * 0.5]
    x = np.concatenate(rows)
    xb = _bits(x)
    codes, params = oracle.quantize_q3(xb)
    xv = oracle.bf16_to_f64(xb)
    n_rows, D = xv.shape
    q = oracle.q3_code_values(codes, D)
    slack = Fraction(8 * 3, 2 ** 24)
    n_codes = n_diff = n_param_diff = 0
    for r in range(n_rows):
        for grp in range(D // 32):
            vals = [Fraction(float(v)) for v in xv[r, 32 * grp: 32 * grp + 32]]
            mn, mx = min(vals), max(vals)
            s_ex = _fp16_round_exact((mx - mn) / 7)
            z_ex = _fp16_round_exact(mn)
            s_got, z_got = params[r, 2 * grp], params[r, 2 * grp + 1]
            assert z_got == z_ex, (r, grp)
            if s_got != s_ex:
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
                exact = min(7, max(0, round(t)))
                if got != exact:
                    n_diff += 1
                    half = Fraction(2 * min(got, exact) + 1, 2)
                    assert abs(got - exact) == 1 and abs(t - half) <= slack, (r, grp, d, float(t))
    assert n_codes == n_rows * D
    assert n_diff <= n_codes // 10000, n_diff
    assert n_param_diff <= (n_rows * D // 32) // 1000, n_param_diff
    print(f"exact-rounding pin: {n_diff} of {n_codes} codes and {n_param_diff} scales differ (all at ties)")
