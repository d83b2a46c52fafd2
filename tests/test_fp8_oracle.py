"""Pins of the FP8 (E4M3) KV oracle (oracle/fp8.py): the code table against
the format's definition, round-to-nearest-even at midpoints, saturation,
underflow, and a brute-force nearest-code check."""
import numpy as np
import pytest

from oracle import fp8
from prefix_shared_kv_radixattention_gb300 import inputs


def test_table_values():
    """Values fixed by the E4M3 layout (bias 7, subnormals m/8 * 2^-6, one
    NaN pattern per sign, no infinities)."""
    t = fp8.decode_table()
    assert t[0x00] == 0.0 and np.signbit(t[0x80]) and t[0x80] == 0.0
    assert t[0x01] == 2.0 ** -9                       # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9                   # largest subnormal
    assert t[0x08] == 2.0 ** -6                       # smallest normal
    assert t[0x38] == 1.0 and t[0x39] == 1.125 and t[0x3F] == 1.875
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0     # largest finite
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)                    # codes 0..126 increase
    assert np.array_equal(t[0x80:0xFF], -pos)          # sign symmetry


def test_exact_values_round_trip():
    t = fp8.decode_table()
    codes = np.array([c for c in range(256) if not np.isnan(t[c])], np.uint8)
    got = fp8.encode(t[codes])
    # every finite code encodes back to itself (-0 keeps its sign)
    assert np.array_equal(got, codes)


def test_ties_to_even_and_rounding():
    # 1.0 (0x38) and 1.125 (0x39): the midpoint goes to the even 0x38
    assert fp8.encode(1.0625) == 0x38
    # 1.125 (0x39) and 1.25 (0x3A): the midpoint goes to 0x3A
    assert fp8.encode(1.1875) == 0x3A
    # off the midpoint, the nearer code
    assert fp8.encode(1.06) == 0x38 and fp8.encode(1.07) == 0x39
    # subnormal spacing 2^-9: 2.5 * 2^-9 ties to 2 * 2^-9 (even), 3.5 to 4
    assert fp8.encode(2.5 * 2 ** -9) == 0x02 and fp8.encode(3.5 * 2 ** -9) == 0x04
    # largest subnormal to smallest normal: 7.5 * 2^-9 ties to 8 * 2^-9 (0x08)
    assert fp8.encode(7.5 * 2 ** -9) == 0x08


def test_saturation_underflow_nan():
    assert fp8.encode(448.0) == 0x7E and fp8.encode(460.0) == 0x7E and fp8.encode(1e30) == 0x7E
    assert fp8.encode(-1e30) == 0xFE
    assert fp8.encode(2.0 ** -10) == 0x00            # half the smallest subnormal: tie to even 0
    assert fp8.encode(1.01 * 2.0 ** -10) == 0x01
    assert fp8.encode(-2.0 ** -11) == 0x80
    assert fp8.encode(np.nan) == 0x7F


def test_brute_force_nearest():
    """On a dense grid over the range: the chosen code's value is at least as
    near as every other finite code's, and on a tie the code is even."""
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(-470, 470, 4000), rng.uniform(-0.02, 0.02, 4000),
                        rng.standard_normal(4000)])
    codes = fp8.encode(x)
    t = fp8.decode_table()
    finite = np.array([c for c in range(256) if not np.isnan(t[c])])
    for xi, c in zip(x, codes):
        if abs(xi) >= 448:
            assert t[c] == np.copysign(448.0, xi)
            continue
        d = np.abs(t[finite] - xi)
        best = d.min()
        assert abs(t[c] - xi) == best
        ties = finite[d == best]
        if len(set(t[ties])) > 1:                     # a true midpoint between two values
            assert c % 2 == 0


def test_quantize_with_scale():
    """A pool scale divides before encoding (in fp32) and multiplies back."""
    x = np.array([0.0, 1.0, -3.0, 100.0, 1e-3], np.float32)
    scale = 0.5
    codes = fp8.quantize_rows(x, scale)
    assert codes.tolist() == fp8.encode(x.astype(np.float64) / scale).tolist()
    back = fp8.dequantize(codes, scale)
    assert back[1] == 1.0 and back[2] == -3.0
    # 100 / 0.5 = 200 lies midway between 192 (mantissa 4) and 208: it rounds
    # to the even 192, read back as 96
    assert back[3] == 96.0
    # relative error of E4M3 is at most 2^-4 for normal values
    xs = np.random.default_rng(1).uniform(0.1, 200.0, 1000).astype(np.float32)
    r = fp8.dequantize(fp8.quantize_rows(xs, 1.0), 1.0)
    assert np.max(np.abs(r - xs) / xs) <= 2.0 ** -4


# ---------------------------------------------------------------------------
# attention over FP8 pools
# ---------------------------------------------------------------------------


def _brute_fp8(q_bits, kc, vc, ks, vs, rtt, row, kend, scale):
    """The definition written out densely in numpy fp64 on the dequantized
    values: softmax over keys 0 .. kend - 1 of the gathered rows."""
    import oracle  # noqa: F401  (package import only)
    qf = inputs.bf16_to_f32(q_bits).astype(np.float64)
    n, hq, d = qf.shape
    hkv = kc.shape[1]
    G = hq // hkv
    o = np.zeros((n, hq, d))
    lse = np.zeros((n, hq))
    for i in range(n):
        slots = rtt[row[i], :kend[i]]
        K = fp8.dequantize(kc[slots], ks)
        V = fp8.dequantize(vc[slots], vs)
        for h in range(hq):
            s = K[:, h // G, :] @ qf[i, h] * scale
            m = s.max()
            w = np.exp(s - m)
            o[i, h] = w @ V[:, h // G, :] / w.sum()
            lse[i, h] = m + np.log(w.sum())
    return o, lse


@pytest.mark.parametrize("ks,vs", [(1.0, 1.0), (0.37, 2.6), (1 / 64, 48.0)])
def test_fp8_attention_is_the_definition_on_dequantized_values(ks, vs):
    rng = np.random.default_rng(int(ks * 1000) + 3)
    S, hkv, hq, d = 40, 2, 4, 16
    kc = rng.integers(0, 0x7F, size=(S, hkv, d)).astype(np.uint8) | (rng.integers(0, 2, size=(S, hkv, d)) << 7).astype(np.uint8)
    vc = rng.integers(0, 0x7F, size=(S, hkv, d)).astype(np.uint8) | (rng.integers(0, 2, size=(S, hkv, d)) << 7).astype(np.uint8)
    kc[kc & 0x7F == 0x7F] = 0                       # no NaN codes
    vc[vc & 0x7F == 0x7F] = 0
    rtt = np.stack([rng.permutation(S)[:24] for _ in range(3)]).astype(np.int32)
    q = inputs.randn_bf16(rng, (5, hq, d))
    row = np.array([0, 1, 2, 0, 2], np.int32)
    kend = np.array([1, 7, 24, 13, 2], np.int32)
    scale = 0.25
    o, lse = fp8.attention(q, kc, vc, ks, vs, rtt, row, np.zeros(5, np.int32), kend, scale)
    bo, blse = _brute_fp8(q, kc, vc, ks, vs, rtt, row, kend, scale)
    assert np.allclose(o, bo, rtol=1e-12, atol=1e-12 * max(1.0, vs))
    assert np.allclose(lse, blse, rtol=1e-12, atol=1e-12)


def test_fp8_bf16_bits_are_exact():
    codes = np.arange(256, dtype=np.uint8)
    finite = ~np.isnan(fp8.decode(codes))
    back = inputs.bf16_to_f32(fp8.bf16_bits(codes)).astype(np.float64)
    assert np.array_equal(back[finite], fp8.decode(codes)[finite])
    assert np.isnan(back[~finite]).all()
