"""Pins of the MLA oracle (CPU): against torch's scaled-dot-product attention
in float64 (multi-query form: one key/value head for every query head, the
values the first dv columns of the keys), closed forms, the empty context,
and the per-token byte counts the pages print."""

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle.kvbytes import kv_bytes_per_token, mla_kv_bytes_per_token
from oracle.mla import mla_decode_attention

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _case(B, Hq, d, S, lens, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, d))
    pool = rng.standard_normal((S, d))
    ld = max(lens) if max(lens) > 0 else 1
    table = np.full((B, ld), -1, dtype=np.int64)
    for r, L in enumerate(lens):
        table[r, :L] = rng.choice(S, size=L, replace=False)
    return q, pool, table, np.asarray(lens)


@pytest.mark.parametrize("Hq,d,dv", [(16, 576, 512), (4, 40, 32), (128, 576, 512)])
def test_mla_equals_sdpa_float64(Hq, d, dv):
    lens = [1, 37, 200]
    q, pool, table, seq = _case(3, Hq, d, 400, lens, seed=Hq + d)
    scale = 1.0 / math.sqrt(192.0)   # a model scale other than the default
    O, L = mla_decode_attention(q, pool, table, seq, dv, sm_scale=scale)
    for r, n in enumerate(lens):
        C = torch.from_numpy(pool[table[r, :n]])                     # [n, d]
        qq = torch.from_numpy(q[r])[None, :, None, :]                # [1, Hq, 1, d]
        kk = C[None, None].expand(1, Hq, n, d)
        vv = C[None, None, :, :dv].expand(1, Hq, n, dv)
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=scale)[0, :, 0]
        assert np.allclose(O[r], ref.numpy(), atol=1e-12)
        lse = torch.logsumexp(scale * (torch.from_numpy(q[r]) @ C.T), dim=1)
        assert np.allclose(L[r], lse.numpy(), atol=1e-12)


def test_mla_identical_rows_closed_form():
    d, dv, n = 576, 512, 50
    rng = np.random.default_rng(3)
    c = rng.standard_normal(d)
    pool = np.tile(c, (n, 1))
    q = rng.standard_normal((1, 2, d))
    table = np.arange(n)[None]
    O, L = mla_decode_attention(q, pool, table, [n], dv)
    for h in range(2):
        assert np.allclose(O[0, h], c[:dv], atol=1e-13)
        assert math.isclose(L[0, h], (q[0, h] @ c) / math.sqrt(d) + math.log(n), rel_tol=0, abs_tol=1e-12)


def test_mla_value_is_the_latent_prefix():
    # one position: the output is exactly that row's first dv elements, not
    # any other window of it
    d, dv = 576, 512
    rng = np.random.default_rng(4)
    pool = rng.standard_normal((2, d))
    q = rng.standard_normal((1, 3, d))
    O, L = mla_decode_attention(q, pool, np.array([[1]]), [1], dv)
    assert np.array_equal(O[0], np.tile(pool[1, :dv], (3, 1)))
    assert np.allclose(L[0], (q[0] @ pool[1]) / math.sqrt(d), atol=1e-13)


def test_mla_empty_context():
    q = np.ones((2, 4, 576))
    table = np.array([[5, 6], [-1, -1]])
    O, L = mla_decode_attention(q, np.ones((8, 576)), table, [2, 0], 512)
    assert np.all(O[1] == 0) and np.all(np.isneginf(L[1])) and np.all(np.isfinite(L[0]))


def test_mla_bytes_per_token_match_the_pages():
    g = json.load(open(os.path.join(GOLDEN, "kv_bytes_mla_deepseek_coder_v2.json")))
    one = mla_kv_bytes_per_token(g["latent_dim"], g["rope_dim"], g["dtype_bytes"])
    assert one == g["mla_bytes_per_token_per_layer"]
    allk = mla_kv_bytes_per_token(g["latent_dim"], g["rope_dim"], g["dtype_bytes"], g["num_layers"]) / 1000
    assert round(allk) == g["mla_bytes_per_token_all_layers_kb_approx"]
    gqa = kv_bytes_per_token(g["gqa_num_kv_heads"], g["gqa_head_dim"], g["dtype_bytes"], g["num_layers"]) / 1000
    assert round(gqa) == g["gqa_bytes_per_token_all_layers_kb_approx"]
