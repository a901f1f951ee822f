"""Pins for the oracle radix cache (oracle/tree.py) -- CPU only.

The trie is checked against things other than itself:
  * a brute-force model that stores every inserted full-page prefix in a hash
    map (the exact-match alternative the bhfrc.com page contrasts with the
    radix tree, §3.1) and computes the longest common prefix by scanning all
    inserted sequences;
  * invariants the pages state: a referenced node is never evicted, eviction
    removes leaves only and in least-recently-used order, cache and requests
    share one pool so slots are conserved;
  * the pages' worked example of three requests sharing a 100-token system
    prompt.
"""

import json
import os
import random

import pytest

from oracle.tree import RadixTrie, NoSlotsError, StateError, build_batch


def _lcp(a, b):
    n = 0
    for x, y in zip(a, b):
        if x != y:
            break
        n += 1
    return n


class BruteCache:
    """Hash map from every inserted full-page prefix to its slots."""

    def __init__(self, P):
        self.P = P
        self.seqs = []
        self.slots_of_prefix = {}

    def insert(self, toks, slots):
        P = self.P
        n_full = len(toks) // P * P
        self.seqs.append(list(toks[:n_full]))
        for k in range(P, n_full + 1, P):
            key = tuple(toks[:k])
            if key not in self.slots_of_prefix:
                self.slots_of_prefix[key] = list(slots[k - P:k])

    def match_len(self, q):
        P = self.P
        q_full = len(q) // P * P
        best = 0
        for s in self.seqs:
            best = max(best, min(_lcp(q, s), q_full, len(s)) // P * P)
        return best

    def match_slots(self, q, m):
        out = []
        for k in range(self.P, m + 1, self.P):
            out.extend(self.slots_of_prefix[tuple(q[:k])])
        return out


@pytest.mark.parametrize("P", [1, 2, 3])
@pytest.mark.parametrize("seed", range(40))
def test_match_equals_bruteforce_lcp(P, seed):
    rnd = random.Random(seed * 7 + P)
    trie = RadixTrie(num_slots=600 * P, page_size=P, free_order=rnd.sample(range(600), 600))
    brute = BruteCache(P)
    for _ in range(60):
        n = rnd.randint(0, 12)
        toks = [rnd.randint(0, 2) for _ in range(n)]
        if rnd.random() < 0.5:
            m, slots, _ = trie.match(toks)
            assert m == brute.match_len(toks)
            assert slots == brute.match_slots(toks, m)
        else:
            rows, lasts, private = build_batch(trie, [toks])
            m_b = brute.match_len(toks)
            assert rows[0][:m_b] == brute.match_slots(toks, m_b)
            brute.insert(toks, rows[0])
            trie.unlock(lasts[0])
            trie.free_slots(private[0])


def test_insert_duplicate_pages_return_to_free_list():
    trie = RadixTrie(num_slots=32, page_size=2, free_order=list(range(16)))
    a = trie.alloc(6)                      # pages 0,1,2
    trie.insert([5, 6, 7, 8, 9, 1], a)
    b = trie.alloc(6)                      # pages 3,4,5
    dup, _ = trie.insert([5, 6, 7, 8, 4, 4], b)
    assert dup == 4                        # two existing pages; caller's pages 3,4 are duplicates
    assert list(trie.free)[-2:] == [3, 4]
    m, slots, _ = trie.match([5, 6, 7, 8, 4, 4])
    assert m == 6 and slots == a[:4] + b[4:]


def test_partial_tail_page_is_never_shared():
    trie = RadixTrie(num_slots=64, page_size=4)
    rows, lasts, private = build_batch(trie, [[1, 2, 3, 4, 5, 6], [1, 2, 3, 4, 5, 6]])
    assert rows[0][:4] == rows[1][:4]
    assert rows[0][4:] != rows[1][4:]
    assert len(private[0]) == 2 and len(private[1]) == 2
    assert trie.tree_tokens() == 4


def _check_conservation(trie, private_total):
    held = trie.tree_tokens() + private_total
    assert len(trie.free) * trie.P + held == trie.num_pages * trie.P


@pytest.mark.parametrize("P", [1, 2])
@pytest.mark.parametrize("seed", range(30))
def test_eviction_invariants(P, seed):
    rnd = random.Random(1000 + seed)
    pages = 24
    trie = RadixTrie(num_slots=pages * P, page_size=P, free_order=rnd.sample(range(pages), pages))
    live = []                  # (last node, private slots)
    for _ in range(80):
        op = rnd.random()
        if op < 0.45:
            toks = [rnd.randint(0, 2) for _ in range(rnd.randint(1, 10))]
            locked_before = {id(n) for n in trie.nodes() if n.ref > 0}
            nodes_before = {id(n): n for n in trie.nodes()}
            try:
                rows, lasts, private = build_batch(trie, [toks])
            except NoSlotsError:
                pass
            else:
                live.append((lasts[0], private[0]))
            now = {id(n) for n in trie.nodes()}
            for k in locked_before:
                assert k in now, "a referenced node was evicted"
        elif op < 0.7 and live:
            last, priv = live.pop(rnd.randrange(len(live)))
            trie.unlock(last)
            trie.free_slots(priv)
        else:
            want = rnd.randint(1, 8)
            before = {id(n): n for n in trie.nodes()}
            freed = trie.evict(want)
            after = {id(n) for n in trie.nodes()}
            gone = [before[k] for k in before if k not in after]
            assert freed == len(gone) * trie.P
            assert all(n.ref == 0 for n in gone), "a referenced node was evicted"
            # prefix-closed: every surviving node's parent survives (leaves go first)
            for k in after:
                p = before[k].parent
                assert p is trie.root or id(p) in after
            # least recently used first: a parent is stamped whenever a child
            # is, so no surviving unreferenced leaf is older than an evicted node
            if gone:
                newest_gone = max(n.last_access for n in gone)
                for n in trie.nodes():
                    if not n.children and n.ref == 0:
                        assert n.last_access >= newest_gone
            if freed < want:
                assert not any(not n.children and n.ref == 0 for n in trie.nodes()), "stopped early"
        _check_conservation(trie, sum(len({s // trie.P for s in p}) * trie.P for _, p in live))


def test_eviction_order_is_lru_on_a_fixed_history():
    # three independent sequences touched at known times; the oldest goes first
    trie = RadixTrie(num_slots=12, page_size=1, free_order=list(range(12)))
    for toks in ([0, 0], [1, 1], [2, 2]):
        rows, lasts, _ = build_batch(trie, [toks])
        trie.unlock(lasts[0])
    trie.match([0, 0])                     # [0,0] is now the most recent
    assert trie.evict(2) == 2
    assert trie.match([1, 1])[0] == 0      # [1,1] was least recently used
    assert trie.match([0, 0])[0] == 2 and trie.match([2, 2])[0] == 2


def test_locked_path_survives_full_eviction_and_unlock_underflow_errors():
    trie = RadixTrie(num_slots=8, page_size=1)
    rows, lasts, _ = build_batch(trie, [[1, 2, 3]])
    assert trie.evict(100) == 0
    trie.unlock(lasts[0])
    with pytest.raises(StateError):
        trie.unlock(lasts[0])
    assert trie.evict(100) == 3


def test_pool_exhaustion_raises_and_releases_locks():
    trie = RadixTrie(num_slots=8, page_size=1)
    with pytest.raises(NoSlotsError):
        build_batch(trie, [[1, 2, 3, 4, 5], [7, 8, 9, 9]])
    assert all(n.ref == 0 for n in trie.nodes())
    assert trie.evict(100) == 5


def test_worked_example_shared_system_prompt(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "shared_system_prompt_3_requests.json")))
    sys_toks = list(range(1000, 1000 + g["shared_system_tokens"]))
    users = [[5, 6, 7], [8, 9, 10, 11], [12, 13]]
    trie = RadixTrie(num_slots=1024, page_size=1)
    rows, _, _ = build_batch(trie, [sys_toks + u for u in users[:g["requests"]]])
    uniq = sum(len(u) for u in users)
    assert trie.tree_tokens() == g["shared_system_kv_tokens"] + uniq
    unshared = g["requests"] * g["shared_system_tokens"] + uniq
    assert unshared - trie.tree_tokens() == g["saved_kv_tokens"]
    assert rows[0][:100] == rows[1][:100] == rows[2][:100]
