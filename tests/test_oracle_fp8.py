"""Pins of the oracle's E4M3 encoder and FP8 KV write (no GPU).

The encoder is the format's definition (nearest finite value, ties to the
even mantissa, saturation to 448, NaN kept); it is pinned against torch's
float8_e4m3fn conversion wherever the two readings agree (below the
saturation point, where torch returns NaN instead), against closed forms,
and against planted mistakes that each of those catches.
"""

import numpy as np
import torch

from oracle.fp8 import e4m3_to_float, float_to_e4m3, kv_write_e4m3, quantise_rows


def _all_finite_bf16():
    bits = np.arange(65536, dtype=np.uint32) << 16
    f = bits.view(np.float32)
    return f[np.isfinite(f)]


def test_encoding_equals_torch_below_saturation():
    f = _all_finite_bf16()
    rng = np.random.default_rng(5)
    f = np.concatenate([f, rng.standard_normal(200000).astype(np.float32) * np.float32(50)])
    f = f[np.abs(f) < 464]
    ref = torch.from_numpy(f.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(float_to_e4m3(f.astype(np.float64)), ref)


def test_encoding_closed_forms():
    # every finite code is its own nearest value (both signs, both zeros)
    codes = np.arange(256, dtype=np.uint8)
    fin = ~np.isnan(e4m3_to_float(codes))
    assert np.array_equal(float_to_e4m3(e4m3_to_float(codes[fin])), codes[fin])
    # ties go to the even mantissa: 1.0625 between 1 (0x38) and 1.125 (0x39),
    # 1.1875 between 1.125 and 1.25 (0x3A); 2^-10 between 0 and 2^-9 (0x01)
    assert list(float_to_e4m3([1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -11])) == [0x38, 0x3A, 0x00, 0x01]
    # saturation to 448 with the sign; NaN stays NaN
    assert list(float_to_e4m3([448.0, 460.0, 464.0, 1e9, -1e9, np.inf])) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7E]
    assert float_to_e4m3([np.nan])[0] & 0x7F == 0x7F


def test_planted_encoder_mistakes_are_caught():
    f = _all_finite_bf16()
    f = f[np.abs(f) < 464].astype(np.float64)
    ref = torch.from_numpy(f.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    vals = e4m3_to_float(np.arange(0x7F))

    def nearest(x, tie):   # nearest finite code, `tie` choosing between (lo, hi)
        a = np.abs(x)
        hi = np.minimum(np.searchsorted(vals, a), 0x7E)
        lo = np.maximum(hi - 1, 0)
        dl, dh = a - vals[lo], vals[hi] - a
        c = np.where(dh < dl, hi, np.where(dl < dh, lo, tie(lo, hi)))
        c = np.where(a >= 448.0, 0x7E, c)
        return (c | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)

    assert np.array_equal(nearest(f, lambda lo, hi: np.where(hi % 2 == 0, hi, lo)), ref)   # the definition
    mistakes = {
        "ties away from zero": lambda x: nearest(x, lambda lo, hi: hi),
        "ties toward zero": lambda x: nearest(x, lambda lo, hi: lo),
        "truncation": lambda x: np.where(np.abs(e4m3_to_float(float_to_e4m3(x))) > np.abs(x),
                                         float_to_e4m3(x) - 1, float_to_e4m3(x)).astype(np.uint8),
        "subnormals flushed": lambda x: np.where((float_to_e4m3(x) & 0x78) == 0, float_to_e4m3(x) & 0x80,
                                                 float_to_e4m3(x)).astype(np.uint8),
    }
    for name, bad in mistakes.items():
        assert not np.array_equal(bad(f), ref), name


def test_quotient_is_taken_in_float32():
    # 1.5 / 3 in float32 and float64 differ in their last bits but encode the
    # same; a value whose float32 quotient lands exactly on a tie shows the
    # single float32 rounding: x = 3 * 1.0625 / 3 == 1.0625 exactly in float32
    x = np.array([3.1875], dtype=np.float32)    # 3 * 1.0625
    assert quantise_rows(x, 3.0)[0] == 0x38     # 1.0625 -> tie -> even (1.0)
    assert quantise_rows(np.array([0.0], dtype=np.float32), 0.5)[0] == 0


def test_kv_write_e4m3_stores_codes_at_their_slots_only():
    rng = np.random.default_rng(2)
    S, Hkv, d = 64, 2, 16
    kc = rng.integers(0, 256, size=(S, Hkv, d), dtype=np.uint8)
    vc = rng.integers(0, 256, size=(S, Hkv, d), dtype=np.uint8)
    k0, v0 = kc.copy(), vc.copy()
    table = np.array([[5, 9, 11, 40], [7, 8, 30, 31]], dtype=np.int64)
    pre, ext = [1, 2], [3, 2]
    kn = rng.standard_normal((5, Hkv, d)).astype(np.float32)
    vn = rng.standard_normal((5, Hkv, d)).astype(np.float32)
    kv_write_e4m3(kc, vc, kn, vn, 0.25, 0.5, table, pre, ext)
    written = [9, 11, 40, 30, 31]
    for i, sl in enumerate(written):
        assert np.array_equal(kc[sl], quantise_rows(kn[i], 0.25))
        assert np.array_equal(vc[sl], quantise_rows(vn[i], 0.5))
    rest = np.setdiff1d(np.arange(S), written)
    assert np.array_equal(kc[rest], k0[rest]) and np.array_equal(vc[rest], v0[rest])
