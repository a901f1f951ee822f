"""Oracle MLA decode attention (latent space, after weight absorption), in
float64.

Test infrastructure only (see ``oracle/__init__``).

Source (page title, section): the CS349D lecture-16 notes (SGLang case
study), §4 "More engineering" (kernels and compilation: for DeepSeek's MLA
the decompression matrices are absorbed into the query and output
projections and attention runs directly in the 576-dimensional latent
space, with a grouped decode kernel) and §5.1 "DP attention" (MLA stores per
token one 512-dimensional latent vector plus a 64-dimensional position part,
1,152 bytes per token and layer in bf16, and has a single KV "head" that all
query heads read).

Definitions (with the readings taken): per token the pool holds ONE
row ``c`` of ``d = 576`` elements (latent first, then the position part).
For request r and query head h (every head reads the same row):
  s_j  = sm_scale * <q[r, h], c[slot(r, j)]>           (all 576 elements)
  LSE  = m + ln sum_j exp(s_j - m),  m = max_j s_j      (natural log)
  O    = sum_j exp(s_j - LSE) * c[slot(r, j)][:dv]      (dv = 512: the latent)
with sm_scale = 1/sqrt(d) unless given (the model's own scale is a
parameter).  An empty context gives O = 0, LSE = -inf.  No sharing is used.
"""

import math

import numpy as np


def mla_decode_attention(q, kv_pool, req_to_token, seq_lens, dv, sm_scale=None, requests=None):
    """q [B, Hq, d]; kv_pool [S, d] (anything whose ``[slots]`` gives float
    rows); req_to_token [B, ld]; seq_lens [B].  Returns O [B, Hq, dv] and
    LSE [B, Hq] (float64); with ``requests`` only those rows are computed."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    table = np.asarray(req_to_token)
    lens = np.asarray(seq_lens)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    O = np.zeros((B, Hq, dv))
    LSE = np.full((B, Hq), -math.inf)
    for r in (range(B) if requests is None else requests):
        r = int(r)
        L = int(lens[r])
        if L == 0:
            continue
        C = np.asarray(kv_pool[np.asarray(table[r, :L], dtype=np.int64)], dtype=np.float64).reshape(L, d)
        for h in range(Hq):
            s = sm_scale * (C @ q[r, h])
            m = s.max()
            w = np.exp(s - m)
            l = w.sum()
            LSE[r, h] = m + math.log(l)
            O[r, h] = (w / l) @ C[:, :dv]
    return O, LSE
