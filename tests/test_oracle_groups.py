"""Pins for the oracle prefix groups (oracle/groups.py) -- CPU only.

  * the vectorised definition equals the pure-Python transcription of the
    definition on random batches built by the oracle trie (page sizes 1-3,
    identical requests, requests that are prefixes of others, empty ones);
  * the batch whose requests end at every node of the conversation-tree
    figure on the chenxutan.com page yields exactly the figure's nodes;
  * every position of every request is covered by exactly one of its
    segments, and all members read the same slots there.
"""

import json
import os
import random

import numpy as np
import pytest

from oracle.groups import prefix_groups, prefix_groups_bruteforce
from oracle.tree import RadixTrie, build_batch


def _table(rows):
    B = len(rows)
    ld = max([len(r) for r in rows] + [1])
    t = np.full((B, ld), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        t[i, :len(r)] = r
    return t, np.array([len(r) for r in rows], dtype=np.int32)


def _same(a, b):
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def _random_batch(rnd, P):
    trie = RadixTrie(num_slots=4096 * P, page_size=P, free_order=rnd.sample(range(4096), 4096))
    # warm the cache with some history, then build a batch
    for _ in range(rnd.randint(0, 4)):
        toks = [rnd.randint(0, 2) for _ in range(rnd.randint(0, 14))]
        _, lasts, priv = build_batch(trie, [toks])
        trie.unlock(lasts[0])
        trie.free_slots(priv[0])
    batch = []
    for _ in range(rnd.randint(1, 7)):
        c = rnd.random()
        if batch and c < 0.2:
            batch.append(list(batch[rnd.randrange(len(batch))]))             # identical request
        elif batch and c < 0.35:
            src = batch[rnd.randrange(len(batch))]
            batch.append(src[:rnd.randint(0, len(src))])                     # a prefix of another
        else:
            batch.append([rnd.randint(0, 2) for _ in range(rnd.randint(0, 14))])
    rows, _, _ = build_batch(trie, batch)
    return rows


@pytest.mark.parametrize("P", [1, 2, 3])
@pytest.mark.parametrize("seed", range(60))
def test_vectorised_groups_equal_definition(P, seed):
    rows = _random_batch(random.Random(seed * 31 + P), P)
    t, lens = _table(rows)
    _same(prefix_groups(t, lens), prefix_groups_bruteforce(rows))


@pytest.mark.parametrize("seed", range(20))
def test_segments_cover_each_request_once(seed):
    rows = _random_batch(random.Random(500 + seed), 1 + seed % 3)
    t, lens = _table(rows)
    g = prefix_groups(t, lens)
    cover = [np.zeros(len(r), dtype=int) for r in rows]
    for s in range(len(g["seg_begin"])):
        b, e, rep = g["seg_begin"][s], g["seg_end"][s], g["seg_row"][s]
        mem = g["seg_members"][g["seg_member_ptr"][s]:g["seg_member_ptr"][s + 1]]
        assert rep == mem.min() and b < e
        for m in mem:
            cover[m][b:e] += 1
            assert list(rows[m][b:e]) == list(rows[rep][b:e])
    for c in cover:
        assert np.all(c == 1)


def test_conversation_tree_figure(golden_dir):
    fig = json.load(open(os.path.join(golden_dir, "conversation_tree_figure.json")))
    nodes = fig["nodes"]
    rnd = random.Random(7)
    toks = {}
    used_first = {}
    for name, spec in nodes.items():          # parents precede children in the file
        first = rnd.randint(0, 10 ** 6)
        while first in used_first.get(spec["parent"], set()):
            first = rnd.randint(0, 10 ** 6)
        used_first.setdefault(spec["parent"], set()).add(first)
        toks[name] = [first] + [rnd.randint(0, 10 ** 6) for _ in range(spec["len"] - 1)]

    def path(name):
        out = []
        while name is not None:
            out.insert(0, name)
            name = nodes[name]["parent"]
        return out

    names = list(nodes)
    batch = [sum((toks[n] for n in path(name)), []) for name in names]
    trie = RadixTrie(num_slots=256, page_size=1)
    rows, _, _ = build_batch(trie, batch)
    g = prefix_groups(*_table(rows))
    got = set()
    for s in range(len(g["seg_begin"])):
        mem = tuple(g["seg_members"][g["seg_member_ptr"][s]:g["seg_member_ptr"][s + 1]])
        got.add((int(g["seg_end"][s] - g["seg_begin"][s]), mem))
    want = set()
    for name in names:
        members = tuple(i for i, other in enumerate(names) if name in path(other))
        want.add((nodes[name]["len"], members))
    assert got == want
    assert len(g["seg_begin"]) == len(names)
