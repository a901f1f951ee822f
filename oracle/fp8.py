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
