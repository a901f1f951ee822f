"""Pins for the oracle attention (oracle/attention.py) and KV-byte formula -- CPU only.

  * closed forms: one key gives O = V and LSE = sm_scale * q.k exactly; all
    logits equal (q = 0) gives O = mean(V) and LSE = ln n;
  * library special cases: torch's scaled_dot_product_attention in float64
    on explicitly gathered K/V (with ``enable_gqa`` fixing the query-head to
    KV-head grouping independently), and scipy's logsumexp for LSE;
  * "compute once, reference many": the shared-aware decode equals the
    unshared decode; splitting every segment into chunks and merging by LSE
    equals the unsplit result (to 1e-12 in float64);
  * extend with no cached prefix is causal attention; extend of one token
    after a prefix is decode;
  * the KV write stores each new row at its slot and nothing else (brute
    force); a prompt prefilled chunk by chunk with the write fused in equals
    causal SDPA over the whole prompt, and its last token equals decode;
  * the worked KV-byte example on the chenxutan.com page.
"""

import json
import math
import os
import random

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

from oracle.attention import (decode_attention, decode_attention_shared, extend_attention,
                              extend_attention_kvwrite, kv_write, lse_merge, softmax_attend)
from oracle.groups import prefix_groups
from oracle.kvbytes import kv_bytes_per_token, unique_kv_bytes, unshared_kv_bytes
from oracle.tree import RadixTrie, build_batch


def _pool(S, Hkv, d, seed):
    g = np.random.default_rng(seed)
    return g.standard_normal((S, Hkv, d)), g.standard_normal((S, Hkv, d))


def _table(rows):
    ld = max([len(r) for r in rows] + [1])
    t = np.full((len(rows), ld), -1, dtype=np.int64)
    for i, r in enumerate(rows):
        t[i, :len(r)] = r
    return t, np.array([len(r) for r in rows])


def test_single_key_closed_form():
    rng = np.random.default_rng(0)
    q, k, v = rng.standard_normal(64), rng.standard_normal((1, 64)), rng.standard_normal((1, 64))
    o, lse = softmax_attend(q, k, v, 0.125)
    assert np.array_equal(o, v[0])
    assert lse == pytest.approx(0.125 * float(q @ k[0]), abs=1e-15)


def test_uniform_logits_closed_form():
    rng = np.random.default_rng(1)
    K, V = rng.standard_normal((37, 32)), rng.standard_normal((37, 32))
    o, lse = softmax_attend(np.zeros(32), K, V, 0.3)
    assert np.allclose(o, V.mean(0), atol=1e-14)
    assert lse == pytest.approx(math.log(37), abs=1e-14)


def test_empty_context():
    o, lse = softmax_attend(np.ones(8), np.zeros((0, 8)), np.zeros((0, 8)), 1.0)
    assert np.all(o == 0) and lse == -math.inf


@pytest.mark.parametrize("Hq,Hkv,d", [(4, 2, 64), (32, 8, 128), (8, 8, 16), (8, 1, 32)])
def test_decode_equals_sdpa_float64(Hq, Hkv, d):
    rng = np.random.default_rng(Hq * 100 + d)
    S, B = 300, 5
    K, V = _pool(S, Hkv, d, 3)
    rows = [list(rng.permutation(S)[:rng.integers(1, 120)]) for _ in range(B)]
    t, lens = _table(rows)
    q = rng.standard_normal((B, Hq, d))
    O, LSE = decode_attention(q, K, V, t, lens)
    scale = 1 / math.sqrt(d)
    for r in range(B):
        kk = torch.from_numpy(K[rows[r]]).permute(1, 0, 2)[None]       # [1, Hkv, L, d]
        vv = torch.from_numpy(V[rows[r]]).permute(1, 0, 2)[None]
        qq = torch.from_numpy(q[r])[None, :, None, :]                    # [1, Hq, 1, d]
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=scale, enable_gqa=True)
        assert np.allclose(O[r], ref[0, :, 0].numpy(), atol=1e-12)
        # LSE from an independent score computation (repeat_interleave grouping)
        kg = torch.from_numpy(K[rows[r]]).repeat_interleave(Hq // Hkv, dim=1)   # [L, Hq, d]
        s = np.einsum("hd,lhd->hl", q[r], kg.numpy()) * scale
        assert np.allclose(LSE[r], logsumexp(s, axis=1), atol=1e-12)


def _shared_batch(seed, P=1):
    rnd = random.Random(seed)
    trie = RadixTrie(num_slots=2048 * P, page_size=P, free_order=rnd.sample(range(2048), 2048))
    prefix = [rnd.randint(0, 50) for _ in range(rnd.randint(1, 40))]
    batch = []
    for _ in range(rnd.randint(2, 6)):
        fork = prefix[:rnd.randint(0, len(prefix))]
        batch.append(fork + [rnd.randint(0, 50) for _ in range(rnd.randint(0, 25))])
    batch.append(list(batch[0]))
    rows, _, _ = build_batch(trie, batch)
    return rows


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("P", [1, 4])
def test_shared_equals_unshared_and_split_invariance(seed, P):
    rows = _shared_batch(seed, P)
    t, lens = _table(rows)
    g = prefix_groups(t, lens)
    Hq, Hkv, d = 8, 2, 16
    K, V = _pool(2048 * P, Hkv, d, seed)
    q = np.random.default_rng(seed).standard_normal((len(rows), Hq, d))
    O0, L0 = decode_attention(q, K, V, t, lens)
    O1, L1 = decode_attention_shared(q, K, V, t, lens, g)
    assert np.allclose(O0, O1, atol=1e-12) and np.allclose(L0, L1, atol=1e-12)
    for chunk in (1, 3, 7):
        O2, L2 = decode_attention_shared(q, K, V, t, lens, g, chunk=chunk)
        assert np.allclose(O0, O2, atol=1e-12) and np.allclose(L0, L2, atol=1e-12)


def test_lse_merge_closed_form():
    rng = np.random.default_rng(5)
    K, V, q = rng.standard_normal((50, 8)), rng.standard_normal((50, 8)), rng.standard_normal(8)
    whole = softmax_attend(q, K, V, 0.5)
    cuts = [0, 1, 17, 18, 50]
    parts = [softmax_attend(q, K[a:b], V[a:b], 0.5) for a, b in zip(cuts[:-1], cuts[1:])]
    parts.append((np.zeros(8), -math.inf))                  # an empty split contributes nothing
    o, lse = lse_merge(parts)
    assert np.allclose(o, whole[0], atol=1e-13)
    assert lse == pytest.approx(logsumexp(0.5 * (K @ q)), abs=1e-13)
    assert lse_merge([(np.zeros(8), -math.inf)])[1] == -math.inf


def test_lse_merge_of_nothing_is_the_empty_context():
    """No partials at all is an empty key set: O = 0 and LSE = -inf, like an
    empty context."""
    o, lse = lse_merge([], d=8)
    assert lse == -math.inf and o.shape == (8,) and not o.any()
    o, lse = lse_merge([])
    assert lse == -math.inf and o.shape == (0,)


def test_extend_no_prefix_is_causal_sdpa():
    rng = np.random.default_rng(9)
    Hq, Hkv, d, S = 8, 2, 32, 512
    K, V = _pool(S, Hkv, d, 4)
    ext = [17, 1, 40]
    rows = [list(rng.permutation(S)[:n]) for n in ext]
    t, _ = _table(rows)
    q = rng.standard_normal((sum(ext), Hq, d))
    O, LSE = extend_attention(q, K, V, t, [0, 0, 0], ext)
    o0 = 0
    for r, n in enumerate(ext):
        qq = torch.from_numpy(q[o0:o0 + n]).permute(1, 0, 2)[None]
        kk = torch.from_numpy(K[rows[r]]).permute(1, 0, 2)[None]
        vv = torch.from_numpy(V[rows[r]]).permute(1, 0, 2)[None]
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, is_causal=True,
                                                               scale=1 / math.sqrt(d), enable_gqa=True)
        assert np.allclose(O[o0:o0 + n], ref[0].permute(1, 0, 2).numpy(), atol=1e-12)
        o0 += n


def test_extend_one_token_after_prefix_is_decode():
    rng = np.random.default_rng(11)
    Hq, Hkv, d, S = 8, 4, 16, 256
    K, V = _pool(S, Hkv, d, 6)
    pre = [10, 0, 55]
    rows = [list(rng.permutation(S)[:n + 1]) for n in pre]
    t, lens = _table(rows)
    q = rng.standard_normal((3, Hq, d))
    Oe, Le = extend_attention(q, K, V, t, pre, [1, 1, 1])
    Od, Ld = decode_attention(q, K, V, t, lens)
    assert np.allclose(Oe, Od, atol=1e-14) and np.allclose(Le, Ld, atol=1e-14)


def test_attention_is_invariant_to_where_slots_live():
    rng = np.random.default_rng(12)
    K, V = _pool(64, 2, 8, 7)
    q = rng.standard_normal((1, 4, 8))
    row = list(rng.permutation(64)[:30])
    perm = rng.permutation(64)
    inv = np.argsort(perm)
    O0, L0 = decode_attention(q, K, V, *_table([row]))
    O1, L1 = decode_attention(q, K[perm], V[perm], *_table([[int(inv[s]) for s in row]]))
    assert np.allclose(O0, O1, atol=1e-14) and np.allclose(L0, L1, atol=1e-14)


def test_kv_bytes_worked_example(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "kv_bytes_llama31_70b.json")))
    per = kv_bytes_per_token(g["num_kv_heads"], g["head_dim"], g["dtype_bytes"], g["num_layers"])
    assert per == g["bytes_per_token"]
    assert per * g["prompt_tokens"] == g["prompt_bytes_gib"] * 2 ** 30


def test_unique_vs_unshared_bytes():
    rows = _shared_batch(3)
    t, lens = _table(rows)
    g = prefix_groups(t, lens)
    distinct = len({s for r in rows for s in r})
    assert unique_kv_bytes(g, 8, 128, 2) == distinct * 4096
    assert unshared_kv_bytes(lens, 8, 128, 2) == sum(len(r) for r in rows) * 4096


def test_kv_write_stores_each_row_at_its_slot_only():
    rng = np.random.default_rng(21)
    S, Hkv, d = 96, 2, 4
    K0, V0 = _pool(S, Hkv, d, 8)
    pre, ext = [3, 0, 7], [5, 2, 1]
    perm = rng.permutation(S)
    rows = [list(perm[0:8]), list(perm[8:10]), list(perm[10:18])]
    t, _ = _table(rows)
    kn = rng.standard_normal((sum(ext), Hkv, d))
    vn = rng.standard_normal((sum(ext), Hkv, d))
    K, V = kv_write(K0.copy(), V0.copy(), kn, vn, t, pre, ext)
    written = {}
    row = 0
    for r in range(3):
        for i in range(ext[r]):
            written[int(t[r, pre[r] + i])] = row
            row += 1
    for slot in range(S):
        if slot in written:
            assert np.array_equal(K[slot], kn[written[slot]]) and np.array_equal(V[slot], vn[written[slot]])
        else:
            assert np.array_equal(K[slot], K0[slot]) and np.array_equal(V[slot], V0[slot])


def test_chunked_prefill_with_kv_write_is_causal_sdpa_and_ends_in_decode():
    rng = np.random.default_rng(22)
    Hq, Hkv, d, S = 4, 2, 16, 300
    K, V = _pool(S, Hkv, d, 9)          # stale contents at the prompt's slots
    L = 70
    slots = list(rng.permutation(S)[:L])
    t, _ = _table([slots])
    q = rng.standard_normal((L, Hq, d))
    kn = rng.standard_normal((L, Hkv, d))
    vn = rng.standard_normal((L, Hkv, d))
    O = np.zeros((L, Hq, d))
    LSE = np.zeros((L, Hq))
    Kc, Vc = K.copy(), V.copy()
    for c0 in range(0, L, 16):          # chunks of 16 new tokens on top of the cached ones
        n = min(16, L - c0)
        O[c0:c0 + n], LSE[c0:c0 + n] = extend_attention_kvwrite(q[c0:c0 + n], kn[c0:c0 + n], vn[c0:c0 + n], Kc, Vc,
                                                                 t, [c0], [n])
        kv_write(Kc, Vc, kn[c0:c0 + n], vn[c0:c0 + n], t, [c0], [n])   # the cache after the chunk
    qq = torch.from_numpy(q).permute(1, 0, 2)[None]
    kk = torch.from_numpy(kn).permute(1, 0, 2)[None]
    vv = torch.from_numpy(vn).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, is_causal=True, scale=1 / math.sqrt(d),
                                                           enable_gqa=True)
    assert np.allclose(O, ref[0].permute(1, 0, 2).numpy(), atol=1e-12)
    Od, Ld = decode_attention(q[L - 1:L], Kc, Vc, t, [L])
    assert np.allclose(O[L - 1:L], Od, atol=1e-13) and np.allclose(LSE[L - 1:L], Ld, atol=1e-13)


def test_e4m3_decoding_equals_torch_for_all_codes():
    from oracle.fp8 import e4m3_to_float
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3_to_float(codes)
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.array_equal(both_nan, np.isnan(ref)) and np.array_equal(got[~both_nan], ref[~both_nan])
    # closed forms: largest finite 448, smallest subnormal 2^-9, one = 0x38
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0 and got[0xB8] == -1.0
