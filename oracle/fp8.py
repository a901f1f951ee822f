"""FP8 E4M3 decoding for the oracle (the FP8 KV cache variant).

Test infrastructure only (see ``oracle/__init__``).

The pages say only that an FP8 KV cache halves the KV bytes ("SGLang 深度拆解",
KV-cache compression with FP8; CS349D lecture-16 notes §4, FP8 KV cache).
Reading: E4M3 as in the OCP 8-bit floating point format -- 1 sign bit, 4
exponent bits with bias 7, 3 mantissa bits; exponent 0 is subnormal
(m / 8 * 2^-6); exponent 15 with mantissa 7 is NaN; there are no infinities
-- and one scale per pool: value = scale * decoded byte.
"""

import numpy as np


def e4m3_to_float(codes):
    """Decode E4M3 bytes (any integer array) to float64."""
    b = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(b >> 7, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    val = np.where(e == 0, sub, normal)
    val = np.where((e == 15) & ((b & 7) == 7), np.nan, val)
    return sign * val


class DequantView:
    """Float64 rows of an FP8 pool (torch uint8 tensor [S, Hkv, d]) times its scale."""

    def __init__(self, tensor, scale):
        self.t = tensor
        self.scale = float(scale)

    def __getitem__(self, slots):
        import torch
        idx = torch.from_numpy(np.asarray(slots, dtype=np.int64))
        return e4m3_to_float(self.t.index_select(0, idx).numpy()) * self.scale


# The 127 non-negative finite codes in increasing order of value (0x00 ..
# 0x7E; 0x7F is NaN): the encoder's candidates.
_FINITE_CODES = np.arange(0x7F, dtype=np.int64)
_FINITE_VALUES = e4m3_to_float(_FINITE_CODES)


def float_to_e4m3(x):
    """Encode values (float64 array) as E4M3 bytes: the nearest finite E4M3
    value, a tie going to the code with an even mantissa; magnitudes beyond
    the largest finite value 448 saturate to it (reading: the write path
    saturates, as a KV cache would rather clip than store NaN); NaN stays
    NaN (0x7F with the sign).  Written as a search over the codes, the
    definition itself."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.int64) << 7
    a = np.abs(x)
    hi = np.searchsorted(_FINITE_VALUES, a, side="left")      # first value >= a
    hi = np.minimum(hi, len(_FINITE_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = np.abs(a - _FINITE_VALUES[lo])
    d_hi = np.abs(_FINITE_VALUES[hi] - a)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((_FINITE_CODES[hi] & 1) == 0))
    code = np.where(pick_hi, _FINITE_CODES[hi], _FINITE_CODES[lo])
    code = np.where(a >= 448.0, 0x7E, code)   # saturation
    code = np.where(np.isnan(x), 0x7F, code)
    return (code | sign).astype(np.uint8)


def quantise_rows(x, scale):
    """E4M3 codes of x / scale with the quotient taken in float32 (IEEE
    division, as the write path computes it), then float_to_e4m3."""
    q = (np.asarray(x, dtype=np.float32) / np.float32(scale)).astype(np.float64)
    return float_to_e4m3(q)


def kv_write_e4m3(k_codes, v_codes, k_new, v_new, k_scale, v_scale, req_to_token, prefix_lens, extend_lens):
    """The KV write into FP8 pools ("SGLang 深度解读", section "5. Attention
    层": the new tokens' K/V go to token_to_kv_pool at their req_to_token
    slots before attention), each stored element the E4M3 code of value /
    scale (quantise_rows).  k_codes, v_codes: uint8 numpy arrays [S, Hkv, d],
    modified in place; k_new, v_new [N, Hkv, d] rows request by request."""
    table = np.asarray(req_to_token)
    kq, vq = quantise_rows(k_new, k_scale), quantise_rows(v_new, v_scale)
    row = 0
    for r in range(len(prefix_lens)):
        pre, ext = int(prefix_lens[r]), int(extend_lens[r])
        for i in range(ext):
            slot = int(table[r, pre + i])
            k_codes[slot] = kq[row]
            v_codes[slot] = vq[row]
            row += 1
    return k_codes, v_codes
