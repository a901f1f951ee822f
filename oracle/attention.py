"""Oracle attention over a slot-indexed KV pool, in float64.

Test infrastructure only (see ``oracle/__init__``).

Sources (page title, section):
  * "SGLang 深度解读" (luoboask.github.io/fde-learning/opensource/sglang/),
    section "5. Attention 层": RadixAttention looks up each request's token
    locations through ``req_to_token`` and reads K/V from the slot-indexed
    ``token_to_kv_pool``; the new tokens' K/V are written to the pool before
    attention runs.
  * "SGLang 深度拆解" (chenxutan.com/d/5669.html) §3.2: decode attends one
    query token to the whole history; prefill/extend attends the uncached
    tokens to the cached prefix plus themselves; scores are scaled by
    1/sqrt(head_dim) and normalised with a softmax (the page's kernels are
    sketches and are not followed; only what they compute is).
  * "SGLang：从前端 DSL 到 SRT 服务运行时", section "用基数树实现前缀复用": a
    shared prefix is computed once and referenced many times -- the basis of
    ``decode_attention_shared``, which must equal ``decode_attention``; and
    its chunked prefill (a long prompt cut into pieces, each prefilled on top
    of the pieces before it) -- the basis of ``extend_attention_kvwrite``
    called chunk by chunk.

Definitions (plain softmax attention, with the readings taken):
  s_j  = sm_scale * <q[r, h], K[slot(r, j), h // G]>,  j < seq_len[r]
  LSE  = m + ln sum_j exp(s_j - m),  m = max_j s_j       (natural log)
  O    = sum_j exp(s_j - LSE) * V[slot(r, j), h // G]
with G = Hq / Hkv (consecutive query heads share a KV head) and
sm_scale = 1/sqrt(d) unless given.  An empty context gives O = 0, LSE = -inf.
"""

import math

import numpy as np


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _rows(pool, slots):
    """Gather pool rows [len(slots), Hkv, d] as float64.

    ``pool`` is any object whose ``__getitem__`` with an int64 index array
    returns the rows (a numpy array or a float64-returning row view).
    """
    slots = np.asarray(slots, dtype=np.int64)
    return _f64(pool[slots])


def softmax_attend(q_vec, K, V, sm_scale):
    """Attention of one query vector over keys K [n, d] and values V [n, d]."""
    n, d = K.shape[0], V.shape[1]
    if n == 0:
        return np.zeros(d), -math.inf
    s = sm_scale * (K @ q_vec)
    m = s.max()
    w = np.exp(s - m)
    l = w.sum()
    lse = m + math.log(l)
    return (w / l) @ V, lse


def decode_attention(q, k_pool, v_pool, req_to_token, seq_lens, sm_scale=None, requests=None):
    """Decode: one query token per request over its whole context.

    q [B, Hq, d]; pools [S, Hkv, d]; req_to_token [B, ld]; seq_lens [B].
    Returns O [B, Hq, d] and LSE [B, Hq] (float64).  No sharing is used.
    With ``requests`` only those rows are computed (others stay 0/-inf).
    """
    q = _f64(q)
    B, Hq, d = q.shape
    table = np.asarray(req_to_token)
    lens = np.asarray(seq_lens)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    O = np.zeros((B, Hq, d))
    LSE = np.full((B, Hq), -math.inf)
    for r in (range(B) if requests is None else requests):
        r = int(r)
        L = int(lens[r])
        K = _rows(k_pool, table[r, :L]) if L else None
        V = _rows(v_pool, table[r, :L]) if L else None
        Hkv = K.shape[1] if L else 1
        G = Hq // Hkv
        for h in range(Hq):
            if L == 0:
                continue
            O[r, h], LSE[r, h] = softmax_attend(q[r, h], K[:, h // G], V[:, h // G], sm_scale)
    return O, LSE


def lse_merge(parts, d=None):
    """Merge partial results [(O_i, LSE_i)] of disjoint key sets into one.

    M = max_i LSE_i;  w_i = exp(LSE_i - M);  O = sum w_i O_i / sum w_i;
    LSE = M + ln sum w_i.  No parts, or only empty ones (LSE -inf), give
    (0, -inf); with no parts at all the zero vector has length ``d`` (0 if
    not given).
    """
    if len(parts) == 0:
        return np.zeros(0 if d is None else d), -math.inf
    lses = np.array([p[1] for p in parts], dtype=np.float64)
    d = len(parts[0][0])
    if np.all(np.isneginf(lses)):
        return np.zeros(d), -math.inf
    M = lses.max()
    w = np.exp(lses - M)
    O = sum(wi * _f64(p[0]) for wi, p in zip(w, parts)) / w.sum()
    return O, M + math.log(w.sum())


def decode_attention_shared(q, k_pool, v_pool, req_to_token, seq_lens, groups,
                            sm_scale=None, chunk=None):
    """Decode that reads every shared segment once and merges by LSE.

    ``groups`` is the prefix-group CSR (see oracle.groups).  For each segment
    [begin, end) the K/V rows of its representative row are gathered ONCE and
    every member's query heads attend to them; each member then merges its
    segments' partials.  ``chunk`` optionally splits every segment further
    into pieces of that many positions (split-KV), which must not change the
    result.
    """
    q = _f64(q)
    B, Hq, d = q.shape
    table = np.asarray(req_to_token)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    parts = [[[] for _ in range(Hq)] for _ in range(B)]
    nseg = len(groups["seg_begin"])
    for s in range(nseg):
        b, e = int(groups["seg_begin"][s]), int(groups["seg_end"][s])
        rep = int(groups["seg_row"][s])
        mem = groups["seg_members"][groups["seg_member_ptr"][s]:groups["seg_member_ptr"][s + 1]]
        step = (e - b) if chunk is None else chunk
        for cb in range(b, e, max(step, 1)):
            ce = min(e, cb + step)
            K = _rows(k_pool, table[rep, cb:ce])
            V = _rows(v_pool, table[rep, cb:ce])
            G = Hq // K.shape[1]
            for r in mem:
                for h in range(Hq):
                    parts[int(r)][h].append(softmax_attend(q[int(r), h], K[:, h // G], V[:, h // G], sm_scale))
    O = np.zeros((B, Hq, d))
    LSE = np.full((B, Hq), -math.inf)
    for r in range(B):
        for h in range(Hq):
            if parts[r][h]:
                O[r, h], LSE[r, h] = lse_merge(parts[r][h])
    return O, LSE


def extend_attention(q_new, k_pool, v_pool, req_to_token, prefix_lens, extend_lens, sm_scale=None,
                     rows=None):
    """Extend (chunked prefill with a cached prefix).

    q_new [N, Hq, d] holds the new tokens of all requests, request by request
    (N = sum extend_lens).  New token i of request r sits at position
    p = prefix_lens[r] + i; its K/V are already in the pool at
    req_to_token[r, p].  It attends to positions 0..p of row r (the cached
    prefix plus the causal part of the new block).
    Returns O [N, Hq, d], LSE [N, Hq].  With ``rows`` (an iterable of
    indices into q_new) only those rows are computed; the others stay 0/-inf.
    """
    q_new = _f64(q_new)
    N, Hq, d = q_new.shape
    table = np.asarray(req_to_token)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    O = np.zeros((N, Hq, d))
    LSE = np.full((N, Hq), -math.inf)
    want = None if rows is None else set(int(x) for x in rows)
    row0 = 0
    for r in range(len(prefix_lens)):
        pre, ext = int(prefix_lens[r]), int(extend_lens[r])
        if ext == 0 or (want is not None and not any(row0 <= x < row0 + ext for x in want)):
            row0 += ext
            continue
        K = _rows(k_pool, table[r, :pre + ext])
        V = _rows(v_pool, table[r, :pre + ext])
        G = Hq // K.shape[1]
        for i in range(ext):
            if want is not None and row0 + i not in want:
                continue
            p = pre + i
            for h in range(Hq):
                O[row0 + i, h], LSE[row0 + i, h] = softmax_attend(
                    q_new[row0 + i, h], K[:p + 1, h // G], V[:p + 1, h // G], sm_scale)
        row0 += ext
    return O, LSE


def kv_write(k_pool, v_pool, k_new, v_new, req_to_token, prefix_lens, extend_lens):
    """Store the new tokens' K/V into the pool ("SGLang 深度解读", section
    "5. Attention 层": K/V go to token_to_kv_pool at their req_to_token slots
    before attention).

    k_pool, v_pool: numpy arrays [S, Hkv, d] (modified in place, any dtype);
    k_new, v_new [N, Hkv, d] rows ordered request by request; new token i of
    request r goes to slot req_to_token[r, prefix_lens[r] + i].
    """
    table = np.asarray(req_to_token)
    row = 0
    for r in range(len(prefix_lens)):
        pre, ext = int(prefix_lens[r]), int(extend_lens[r])
        for i in range(ext):
            slot = int(table[r, pre + i])
            k_pool[slot] = k_new[row]
            v_pool[slot] = v_new[row]
            row += 1
    return k_pool, v_pool


class _Overlay:
    """Rows of ``base`` with some slots replaced (a pool after a KV write,
    without copying the whole pool)."""

    def __init__(self, base, slots, rows):
        self.base = base
        self.new = {int(s): np.asarray(r, dtype=np.float64) for s, r in zip(slots, rows)}

    def __getitem__(self, slots):
        slots = np.asarray(slots, dtype=np.int64)
        out = np.array(_rows(self.base, slots), dtype=np.float64)
        for j, s in enumerate(slots):
            if int(s) in self.new:
                out[j] = self.new[int(s)]
        return out


def extend_attention_kvwrite(q_new, k_new, v_new, k_pool, v_pool, req_to_token, prefix_lens, extend_lens,
                             sm_scale=None, rows=None):
    """Extend with the KV write first: ``kv_write`` of the new rows, then
    ``extend_attention`` over the written pool (the pool itself is not
    modified; the written rows are overlaid)."""
    table = np.asarray(req_to_token)
    slots = []
    for r in range(len(prefix_lens)):
        pre, ext = int(prefix_lens[r]), int(extend_lens[r])
        slots.extend(int(table[r, pre + i]) for i in range(ext))
    kn, vn = _f64(k_new), _f64(v_new)
    return extend_attention(q_new, _Overlay(k_pool, slots, kn), _Overlay(v_pool, slots, vn), table, prefix_lens,
                            extend_lens, sm_scale=sm_scale, rows=rows)
