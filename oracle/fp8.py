"""FP8 (E4M3) key/value storage -- oracle.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.
Plain numpy; it imports nothing from the CUDA path.

The pages do not speak of reduced-precision KV.  FP8 KV is the step beside
the path that a serving deployment takes to halve the bytes decode reads.
The reading taken is the plain one:

* codes are OCP FP8 E4M3 ("fn": no infinities): sign, 4 exponent bits with
  bias 7, 3 mantissa bits.  Exponent field 0 holds the subnormals
  m / 8 * 2^-6; S.1111.111 is NaN; the largest finite value is 448;
* a pool (K or V, per layer) has one fp32 scale: the stored code of x is
  E4M3(x / scale), rounded to the nearest code with ties to the even
  mantissa, magnitudes past 448 saturate to 448, and NaN stays NaN;
* attention over an FP8 pool is the fp64 definition applied to
  decode(code) * scale (``attention``: the bf16-pool oracle on the decoded
  codes, with each pool's scale taken out of its sums).

Pinned in ``tests/test_fp8_oracle.py``.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_NAN = 0x7F


def decode_table() -> np.ndarray:
    """Value of every code 0 .. 255 (float64; NaN for the two NaN codes)."""
    out = np.empty(256, np.float64)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            out[c] = np.nan
        elif e == 0:
            out[c] = sign * (m / 8.0) * 2.0 ** -6
        else:
            out[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


_TABLE = decode_table()
# the finite non-negative codes in value order (0x00 .. 0x7E) and their values
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALUES = _TABLE[:0x7F]


def decode(codes) -> np.ndarray:
    return _TABLE[np.asarray(codes, np.uint8)]


def encode(x) -> np.ndarray:
    """E4M3 codes of float64 values: nearest code, ties to the even mantissa
    (the even code), saturation at 448, NaN to NaN."""
    x = np.asarray(x, np.float64)
    a = np.abs(x)
    # index of the largest positive code value <= a (values are increasing)
    hi_idx = np.searchsorted(_POS_VALUES, np.minimum(a, E4M3_MAX), side="right") - 1
    hi_idx = np.clip(hi_idx, 0, 0x7E)
    lo_val = _POS_VALUES[hi_idx]
    up_idx = np.minimum(hi_idx + 1, 0x7E)
    up_val = _POS_VALUES[up_idx]
    d_lo = a - lo_val
    d_up = up_val - a
    pick_up = (d_up < d_lo) | ((d_up == d_lo) & (up_idx % 2 == 0) & (up_idx != hi_idx))
    code = np.where(pick_up, up_idx, hi_idx)
    code = np.where(a >= E4M3_MAX, 0x7E, code)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), E4M3_NAN, code)
    return code.astype(np.uint8)


def quantize_rows(x, scale: float) -> np.ndarray:
    """Codes of bf16/fp32 values stored with a pool scale: E4M3(x / scale).
    The division is done in fp32, as the store does."""
    y = (np.asarray(x, np.float32) / np.float32(scale)).astype(np.float64)
    return encode(y)


def dequantize(codes, scale: float) -> np.ndarray:
    """The values attention reads from an FP8 pool: decode(code) * scale."""
    return decode(codes) * float(scale)


def bf16_bits(codes) -> np.ndarray:
    """decode(code) as bf16 bits: every E4M3 value (subnormals included) has
    at most 4 significant bits and an exponent inside bf16's range, so the
    float32 of it has 16 zero low bits and the top half is exact."""
    f = decode(codes).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def attention(q, k_codes, v_codes, k_scale: float, v_scale: float, rtt, q_row, kbeg, kend, sm_scale,
              n_threads=None):
    """fp64 attention over FP8 pools: the definition applied to
    decode(code) * scale.  Each pool's scale comes out of its sums:
        s_j = sm_scale * q . (decode(k_j) k_scale) = (sm_scale k_scale) q . decode(k_j),
        o   = sum_j w_j decode(v_j) v_scale / sum_j w_j = v_scale (sum_j w_j decode(v_j) / sum_j w_j),
    so the attention of the decoded codes (exact bf16 values) with the score
    scale sm_scale * k_scale, times v_scale, is that definition.
    Returns (o fp64, lse fp64)."""
    from . import attention as attention_bf16
    o, lse = attention_bf16(q, bf16_bits(k_codes), bf16_bits(v_codes), rtt, q_row, kbeg, kend,
                            float(sm_scale) * float(k_scale), n_threads)
    return o * float(v_scale), lse


def decode_rows(q, k_codes, v_codes, k_scale, v_scale, rtt, req_idx, seq_len, sm_scale, n_threads=None):
    """Decode rows over FP8 pools: one query per request at position L_b - 1."""
    n = len(req_idx)
    return attention(q, k_codes, v_codes, k_scale, v_scale, rtt, np.asarray(req_idx, np.int32),
                     np.zeros(n, np.int32), np.asarray(seq_len, np.int32), sm_scale, n_threads)
