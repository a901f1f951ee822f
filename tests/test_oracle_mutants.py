"""Planted mistakes in the oracle must be caught by its pins -- CPU only.

Each case swaps one oracle function for a copy with one plausible mistake (a
dropped scale, a wrong head mapping, an off-by-one mask, a wrong log base, a
most-recently-used eviction, pages ignored in matching, a merge without
weights, segments not split where a member ends) and checks that at least one
pin test then fails.  Nothing here touches a GPU.
"""

import math

import numpy as np
import pytest

import oracle.attention as OA
import oracle.groups as OG
import oracle.tree as OT
from tests import test_oracle_attention as TA
from tests import test_oracle_groups as TG
from tests import test_oracle_tree as TT


def _fails(fn, *args, **kw):
    try:
        fn(*args, **kw)
    except AssertionError:
        return True
    return False


def test_dropped_softmax_scale_is_caught(monkeypatch):
    good = OA.softmax_attend
    monkeypatch.setattr(OA, "softmax_attend", lambda q, K, V, s: good(q, K, V, 1.0))
    assert _fails(TA.test_decode_equals_sdpa_float64, 4, 2, 64)


def test_log2_lse_is_caught(monkeypatch):
    good = OA.softmax_attend

    def bad(q, K, V, s):
        o, lse = good(q, K, V, s)
        return o, lse / math.log(2)
    monkeypatch.setattr(OA, "softmax_attend", bad)
    monkeypatch.setattr(TA, "softmax_attend", bad)
    assert _fails(TA.test_uniform_logits_closed_form)


def test_wrong_gqa_mapping_is_caught(monkeypatch):
    def bad(q, k_pool, v_pool, req_to_token, seq_lens, sm_scale=None, requests=None):
        q = np.asarray(q, dtype=np.float64)
        B, Hq, d = q.shape
        sm_scale = 1 / math.sqrt(d) if sm_scale is None else sm_scale
        O, L = np.zeros((B, Hq, d)), np.full((B, Hq), -math.inf)
        for r in range(B):
            n = int(seq_lens[r])
            K = np.asarray(k_pool[np.asarray(req_to_token[r, :n])], dtype=np.float64)
            V = np.asarray(v_pool[np.asarray(req_to_token[r, :n])], dtype=np.float64)
            for h in range(Hq):
                O[r, h], L[r, h] = OA.softmax_attend(q[r, h], K[:, h % K.shape[1]], V[:, h % K.shape[1]], sm_scale)
        return O, L
    monkeypatch.setattr(TA, "decode_attention", bad)
    assert _fails(TA.test_decode_equals_sdpa_float64, 32, 8, 128)


def test_causal_off_by_one_is_caught(monkeypatch):
    def bad(q_new, k_pool, v_pool, req_to_token, prefix_lens, extend_lens, sm_scale=None, rows=None):
        # attends to positions 0..p-1 instead of 0..p
        shifted = [max(p - 1, 0) for p in prefix_lens]
        return OA.extend_attention(q_new, k_pool, v_pool, req_to_token, shifted, extend_lens, sm_scale, rows)
    monkeypatch.setattr(TA, "extend_attention", bad)
    assert _fails(TA.test_extend_one_token_after_prefix_is_decode)


def test_unweighted_merge_is_caught(monkeypatch):
    def bad(parts):
        live = [p for p in parts if p[1] != -math.inf]
        return sum(np.asarray(p[0]) for p in live) / len(live), max(p[1] for p in live)
    monkeypatch.setattr(TA, "lse_merge", bad)
    assert _fails(TA.test_lse_merge_closed_form)


def test_mru_eviction_is_caught(monkeypatch):
    def bad_evict(self, num_tokens):
        freed = 0
        while freed < num_tokens:
            cands = self._candidates()
            if not cands:
                break
            victim = max(cands, key=lambda n: (n.last_access, n.nid))
            del victim.parent.children[victim.key]
            self.free.append(victim.page)
            freed += self.P
        return freed
    monkeypatch.setattr(OT.RadixTrie, "evict", bad_evict)
    assert _fails(TT.test_eviction_order_is_lru_on_a_fixed_history)


def test_match_ignoring_pages_is_caught(monkeypatch):
    good = OT.RadixTrie.match

    def bad(self, tokens):
        m, slots, node = good(self, tokens)
        # claims the partial page too when the next page starts the same way
        extra = 0
        child = next((c for k, c in node.children.items() if len(tokens) > m and k[0] == tokens[m]), None)
        if child is not None:
            extra = 1
            slots = slots + [child.page * self.P]
        return m + extra, slots, node
    monkeypatch.setattr(OT.RadixTrie, "match", bad)
    assert any(_fails(TT.test_match_equals_bruteforce_lcp, 2, s) for s in range(10))


def test_segments_not_split_at_member_end_are_caught(monkeypatch):
    def bad(req_to_token, seq_lens):
        # a request that ended stays a member of the segments that continue
        # its path, so groups are not split where a member ends
        rows = [list(req_to_token[i, :int(n)]) for i, n in enumerate(seq_lens)]
        B = len(rows)
        segs = {}
        for r in range(B):
            L, prev, start = len(rows[r]), None, 0
            for j in range(L + 1):
                M = None if j == L else tuple(
                    q for q in range(B) if rows[q][:min(j + 1, len(rows[q]))] == rows[r][:min(j + 1, len(rows[q]))])
                if j > 0 and M != prev:
                    segs[(prev, start)] = j
                    start = j
                prev = M
        return OG._pack(sorted((min(M), b, e, M) for (M, b), e in segs.items()))
    monkeypatch.setattr(TG, "prefix_groups", bad)
    assert _fails(TG.test_conversation_tree_figure, "tests/golden")


def test_kv_write_off_by_one_slot_is_caught(monkeypatch):
    def bad(k_pool, v_pool, k_new, v_new, req_to_token, prefix_lens, extend_lens):
        table = np.asarray(req_to_token)
        row = 0
        for r in range(len(prefix_lens)):
            pre, ext = int(prefix_lens[r]), int(extend_lens[r])
            for i in range(ext):
                slot = int(table[r, max(0, pre + i - 1)])   # one position early
                k_pool[slot] = k_new[row]
                v_pool[slot] = v_new[row]
                row += 1
        return k_pool, v_pool
    monkeypatch.setattr(OA, "kv_write", bad)
    monkeypatch.setattr(TA, "kv_write", bad)
    assert _fails(TA.test_kv_write_stores_each_row_at_its_slot_only)


def test_scheduler_without_deferral_or_with_late_insertion_is_caught(monkeypatch):
    import oracle.sched as OS
    from tests import test_sched as TS
    good = OS.simulate

    def no_defer(trie, requests, **kw):
        kw["defer_tokens"] = 0
        return good(trie, requests, **kw)

    def late_insert(trie, requests, **kw):
        kw["insert_at"] = OS.AT_FINISH
        return good(trie, requests, **kw)
    for bad in (no_defer, late_insert):
        monkeypatch.setattr(TS, "simulate", bad)
        assert _fails(TS.test_few_shot_sharing_needs_insertion_at_prefill)


@pytest.mark.parametrize("mistake", ["bias8", "subnormal_as_normal", "no_sign"])
def test_e4m3_decoding_mistakes_are_caught(monkeypatch, mistake):
    import oracle.fp8 as OF

    def bad(codes):
        b = np.asarray(codes, dtype=np.int64) & 0xFF
        sign = 1.0 if mistake == "no_sign" else np.where(b >> 7, -1.0, 1.0)
        e = (b >> 3) & 0xF
        m = (b & 0x7).astype(np.float64)
        normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - (8.0 if mistake == "bias8" else 7.0))
        sub = normal if mistake == "subnormal_as_normal" else (m / 8.0) * 2.0 ** -6
        val = np.where(e == 0, sub, normal)
        val = np.where((e == 15) & ((b & 7) == 7), np.nan, val)
        return sign * val

    monkeypatch.setattr(OF, "e4m3_to_float", bad)
    assert _fails(TA.test_e4m3_decoding_equals_torch_for_all_codes)


def _mla_mutant(mistake):
    def bad(q, kv_pool, req_to_token, seq_lens, dv, sm_scale=None, requests=None):
        q = np.asarray(q, dtype=np.float64)
        B, Hq, d = q.shape
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(dv if mistake == "scale_by_dv" else d)
        O = np.zeros((B, Hq, dv))
        LSE = np.full((B, Hq), -math.inf)
        for r in range(B):
            L = int(seq_lens[r])
            if L == 0:
                continue
            C = np.asarray(kv_pool[np.asarray(req_to_token[r, :L], dtype=np.int64)], dtype=np.float64).reshape(L, d)
            for h in range(Hq):
                s = sm_scale * (C[:, :dv] @ q[r, h, :dv] if mistake == "latent_only_scores" else C @ q[r, h])
                m = s.max()
                w = np.exp(s - m)
                LSE[r, h] = m + math.log(w.sum())
                V = C[:, d - dv:] if mistake == "value_suffix" else C[:, :dv]
                O[r, h] = (w / w.sum()) @ V
        return O, LSE
    return bad


@pytest.mark.parametrize("mistake", ["scale_by_dv", "latent_only_scores", "value_suffix"])
def test_mla_mistakes_are_caught(monkeypatch, mistake):
    from tests import test_oracle_mla as TM
    monkeypatch.setattr(TM, "mla_decode_attention", _mla_mutant(mistake))
    caught = (_fails(TM.test_mla_equals_sdpa_float64, 16, 576, 512) or _fails(TM.test_mla_identical_rows_closed_form)
              or _fails(TM.test_mla_value_is_the_latent_prefix))
    assert caught
