"""Native host side vs the oracle, bit-exact (CPU).

The C++ compressed radix tree, allocator, batch builder and prefix-group
emitters must reproduce the oracle's per-page trie exactly: match lengths
and slots, duplicate handling, eviction order (observed through the slots
later allocations return), reference counts, req_to_token rows, matched
prefix lengths and prefix groups -- on random operation sequences and on the
five workloads at full size.
"""

import random

import numpy as np
import pytest

import radixattention_prefix_shared_radix_gb300 as sgl
import workloads as W
from oracle.groups import prefix_groups
from oracle.tree import NoSlotsError, RadixTrie, StateError, build_batch
from radixattention_prefix_shared_radix_gb300 import build as sglbuild


@pytest.fixture(scope="module", autouse=True)
def _built():
    sglbuild.build()


def _groups_eq(a, b):
    for k in ("seg_begin", "seg_end", "seg_row", "seg_member_ptr", "seg_members"):
        assert np.array_equal(np.asarray(a[k]), np.asarray(b[k])), k


def _lib_groups(handle):
    return sgl.groups_as_numpy(sgl.sgl_groups_view(handle))


class Pair:
    """The oracle trie and the native tree driven with the same operations."""

    def __init__(self, pages, P, order):
        self.o = RadixTrie(pages * P, P, order)
        self.t = sgl.sgl_tree_create(pages * P, P, order)
        self.P = P
        self.live = []      # (oracle last node, lib last handle, row)

    def close(self):
        sgl.sgl_tree_destroy(self.t)

    def batch(self, seqs):
        try:
            rows, lasts, priv = build_batch(self.o, seqs)
        except NoSlotsError:
            rows = None
        g = sgl.sgl_groups_create()
        try:
            if rows is None:
                with pytest.raises(sgl.SglError) as e:
                    sgl.sgl_build_batch(self.t, seqs, groups=g)
                assert e.value.status == -2
                return
            out = sgl.sgl_build_batch(self.t, seqs, groups=g)
            for r, row in enumerate(rows):
                assert list(out["req_to_token"][r, :len(row)]) == list(row)
                assert np.all(out["req_to_token"][r, len(row):] == -1)
            assert list(out["seq_lens"]) == [len(s) for s in seqs]
            ogroups = prefix_groups(out["req_to_token"], out["seq_lens"])
            _groups_eq(_lib_groups(g), ogroups)
            g2 = sgl.sgl_groups_create()
            sgl.sgl_groups_from_table(out["req_to_token"], out["seq_lens"], g2)
            _groups_eq(_lib_groups(g2), ogroups)
            sgl.sgl_groups_destroy(g2)
            for r in range(len(seqs)):
                self.live.append((lasts[r], int(out["last_nodes"][r]), list(rows[r])))
        finally:
            sgl.sgl_groups_destroy(g)

    def finish(self, k):
        on, ln, row = self.live.pop(k)
        self.o.unlock(on)
        nf = len(row) // self.P * self.P
        self.o.free_slots(row[nf:])
        sgl.sgl_tree_finish(self.t, ln, row, len(row))

    def match(self, toks):
        m, slots, _ = self.o.match(toks)
        m2, slots2, _ = sgl.sgl_tree_match(self.t, toks)
        assert m == m2 and list(slots) == list(slots2)

    def evict(self, n):
        assert self.o.evict(n) == sgl.sgl_tree_evict(self.t, n)

    def alloc_free(self, n):
        try:
            a = self.o.alloc(n)
        except NoSlotsError:
            with pytest.raises(sgl.SglError):
                sgl.sgl_tree_alloc(self.t, n)
            return
        b = sgl.sgl_tree_alloc(self.t, n)
        assert list(a) == list(b)
        self.o.free_slots(a)
        sgl.sgl_tree_free(self.t, b)

    def check_stats(self):
        s = sgl.sgl_tree_stats(self.t)
        assert s["free_pages"] == len(self.o.free)
        assert s["tree_tokens"] == self.o.tree_tokens()
        assert s["locked_tokens"] == sum(self.P for n in self.o.nodes() if n.ref > 0)


@pytest.mark.parametrize("P", [1, 2, 4])
@pytest.mark.parametrize("seed", range(25))
def test_random_operations_bit_exact(P, seed):
    rnd = random.Random(seed * 13 + P)
    pages = rnd.choice([12, 20, 40, 400])
    pair = Pair(pages, P, rnd.sample(range(pages), pages))
    try:
        for _ in range(70):
            op = rnd.random()
            if op < 0.35:
                base = [rnd.randint(0, 2) for _ in range(rnd.randint(0, 10))]
                seqs = []
                for _ in range(rnd.randint(1, 4)):
                    c = rnd.random()
                    if seqs and c < 0.25:
                        seqs.append(list(seqs[0]))
                    else:
                        cut = rnd.randint(0, len(base))
                        seqs.append(base[:cut] + [rnd.randint(0, 2) for _ in range(rnd.randint(0, 8))])
                pair.batch(seqs)
            elif op < 0.55 and pair.live:
                pair.finish(rnd.randrange(len(pair.live)))
            elif op < 0.7:
                pair.match([rnd.randint(0, 2) for _ in range(rnd.randint(0, 12))])
            elif op < 0.85:
                pair.evict(rnd.randint(1, 3 * P))
            else:
                pair.alloc_free(rnd.randint(0, 3 * P))
            pair.check_stats()
    finally:
        pair.close()


def test_unlock_underflow_and_stale_handle():
    t = sgl.sgl_tree_create(16, 1)
    out = sgl.sgl_build_batch(t, [[1, 2, 3]])
    last = int(out["last_nodes"][0])
    sgl.sgl_tree_unlock(t, last)
    with pytest.raises(sgl.SglError) as e:
        sgl.sgl_tree_unlock(t, last)
    assert e.value.status == -6
    assert sgl.sgl_tree_evict(t, 100) == 3
    with pytest.raises(sgl.SglError) as e:
        sgl.sgl_tree_lock(t, last)
    assert e.value.status == -6
    sgl.sgl_tree_destroy(t)


def test_insert_duplicates_match_oracle():
    o = RadixTrie(32, 2, list(range(16)))
    t = sgl.sgl_tree_create(32, 2, list(range(16)))
    for toks in ([5, 6, 7, 8, 9, 1], [5, 6, 7, 8, 4, 4], [5, 6, 7, 8]):
        a = o.alloc(len(toks))
        b = sgl.sgl_tree_alloc(t, len(toks))
        assert list(a) == list(b)
        d1, _ = o.insert(toks, a)
        d2, _ = sgl.sgl_tree_insert(t, toks, b)
        assert d1 == d2
    assert list(o.alloc(16)) == list(sgl.sgl_tree_alloc(t, 16))
    sgl.sgl_tree_destroy(t)


def _full_tables(name):
    w = W.get(name)
    order, _, _ = None, None, None
    S = W.pool_slots(w)
    order = np.random.default_rng([w.seed, 3]).permutation(S // w.page_size).astype(np.int32)
    b = W.make_batch(w)
    o = RadixTrie(S, w.page_size, order)
    t = sgl.sgl_tree_create(S, w.page_size, order)
    if w.kind == "extend":
        warm = [b.cached_tokens(r) for r in range(len(b.req_chain))]
        rows, lasts, _ = build_batch(o, warm)
        for n in lasts:
            o.unlock(n)
        out = sgl.sgl_build_batch(t, warm)
        for r in range(len(warm)):
            sgl.sgl_tree_finish(t, int(out["last_nodes"][r]), out["req_to_token"][r], len(warm[r]))
    return w, b, o, t


@pytest.mark.parametrize("name", ["tiny_fp32", "llama3_8b_decode", "fork_tree", "extend", "multiturn",
                                  "multiturn_noshare"])
def test_workload_tables_bit_exact(name):
    w, b, o, t = _full_tables(name)
    seqs = b.all_tokens()
    rows, _, _ = build_batch(o, seqs)
    g = sgl.sgl_groups_create()
    out = sgl.sgl_build_batch(t, seqs, groups=g)
    table = out["req_to_token"]
    for r, row in enumerate(rows):
        assert np.array_equal(table[r, :len(row)], np.asarray(row, dtype=np.int32))
    if w.kind == "extend":
        assert list(out["prefix_lens"]) == [len(b.cached_tokens(r)) for r in range(len(seqs))]
    _groups_eq(_lib_groups(g), prefix_groups(table, out["seq_lens"]))
    sgl.sgl_groups_destroy(g)
    sgl.sgl_tree_destroy(t)


@pytest.mark.parametrize("P", [1, 4])
def test_finish_batch_equals_finishing_one_by_one(P):
    """sgl_tree_finish_batch leaves the tree exactly as finishing the batch's
    requests one by one does (same stats, same later matches and evictions)."""
    rng = np.random.default_rng(5 + P)
    base = list(rng.integers(0, 1000, size=90))
    seqs = [base + list(rng.integers(0, 1000, size=int(n))) for n in rng.integers(0, 40, size=6)] + [base[:17], []]
    trees = []
    for batched in (False, True):
        t = sgl.sgl_tree_create(4096, P, np.arange(4096 // P, dtype=np.int32))
        out = sgl.sgl_build_batch(t, seqs)
        if batched:
            sgl.sgl_tree_finish_batch(t, out)
        else:
            for r in range(len(seqs)):
                sgl.sgl_tree_finish(t, int(out["last_nodes"][r]), out["req_to_token"][r], len(seqs[r]))
        trees.append(t)
    try:
        assert sgl.sgl_tree_stats(trees[0]) == sgl.sgl_tree_stats(trees[1])
        # the same state: the same eviction, then the same match of every request
        assert sgl.sgl_tree_evict(trees[0], 64) == sgl.sgl_tree_evict(trees[1], 64)
        for s in seqs:
            a, b = sgl.sgl_tree_match(trees[0], s), sgl.sgl_tree_match(trees[1], s)
            assert a[0] == b[0] and np.array_equal(a[1], b[1])
    finally:
        for t in trees:
            sgl.sgl_tree_destroy(t)


def test_build_batch_writes_caller_buffers_in_place():
    """Given output arrays, sgl_build_batch writes the same table and lengths
    into them (and returns them) as into arrays of its own; arrays of the
    wrong type, shape or layout are refused before the tree is touched."""
    import numpy as np
    import radixattention_prefix_shared_radix_gb300 as sgl
    import workloads as W
    w = W.get("llama3_8b_decode_small")
    seqs = W.make_batch(w, 0).all_tokens()
    S = 1 << 14
    ld = max(len(x) for x in seqs) + 3
    trees = [sgl.sgl_tree_create(S, 1, np.arange(S, dtype=np.int32)) for _ in range(2)]
    try:
        for step in range(2):
            a = sgl.sgl_build_batch(trees[0], seqs, ld=ld)
            tab = np.full((len(seqs), ld), 7, dtype=np.int32)
            seq = np.full(len(seqs), 7, dtype=np.int32)
            b = sgl.sgl_build_batch(trees[1], seqs, req_to_token=tab, seq_lens=seq)
            assert b["req_to_token"] is tab and b["seq_lens"] is seq
            for k in ("req_to_token", "seq_lens", "prefix_lens"):
                np.testing.assert_array_equal(a[k], b[k])
            sgl.sgl_tree_finish_batch(trees[0], a)
            sgl.sgl_tree_finish_batch(trees[1], b)
        bad = [dict(req_to_token=np.zeros((len(seqs), ld), dtype=np.int64)),
               dict(req_to_token=np.zeros((len(seqs), ld + 1), dtype=np.int32)[:, :ld]),
               dict(req_to_token=np.zeros((len(seqs) + 1, ld), dtype=np.int32)),
               dict(req_to_token=np.zeros((len(seqs), ld), dtype=np.int32), ld=ld + 1),
               dict(seq_lens=np.zeros(len(seqs) + 1, dtype=np.int32))]
        for kw in bad:
            with pytest.raises(ValueError):
                sgl.sgl_build_batch(trees[1], seqs, **kw)
    finally:
        for t in trees:
            sgl.sgl_tree_destroy(t)


def test_build_batch_from_token_matrix():
    """A [B, cap] token matrix with per-row lengths gives the same tables as
    the list of rows; bad matrices or lengths are refused."""
    import numpy as np
    import radixattention_prefix_shared_radix_gb300 as sgl
    import workloads as W
    w = W.get("fork_tree_small")
    seqs = W.make_batch(w, 0).all_tokens()
    B, cap = len(seqs), max(len(x) for x in seqs) + 5
    mat = np.full((B, cap), 12345, dtype=np.int32)
    for r, x in enumerate(seqs):
        mat[r, :len(x)] = x
    lens = [len(x) for x in seqs]
    S = 1 << 13
    trees = [sgl.sgl_tree_create(S, 1, np.arange(S, dtype=np.int32)) for _ in range(2)]
    try:
        a = sgl.sgl_build_batch(trees[0], seqs, ld=cap)
        b = sgl.sgl_build_batch(trees[1], mat, lens=lens, ld=cap)
        for k in ("req_to_token", "seq_lens", "prefix_lens"):
            np.testing.assert_array_equal(a[k], b[k])
        sgl.sgl_tree_finish_batch(trees[0], a)
        sgl.sgl_tree_finish_batch(trees[1], b)
        # without lens every row is cap tokens long
        full = sgl.sgl_build_batch(trees[1], mat[:2].copy())
        assert list(full["seq_lens"]) == [cap, cap]
        sgl.sgl_tree_finish_batch(trees[1], full)
        for args, kw in [((mat.astype(np.int64),), dict(lens=lens)), ((mat[:, ::2],), dict(lens=lens)),
                         ((mat,), dict(lens=lens[:-1])), ((mat,), dict(lens=[cap + 1] * B)),
                         ((seqs,), dict(lens=lens))]:
            with pytest.raises(ValueError):
                sgl.sgl_build_batch(trees[1], *args, **kw)
    finally:
        for t in trees:
            sgl.sgl_tree_destroy(t)


def _append_run(P, seed, steps):
    """A batch built, advanced `steps` decode steps with sgl_batch_append and
    cached with sgl_tree_cache_finished_batch, against the oracle's
    append_step / cache_finished on the same operations."""
    from oracle.tree import append_step, cache_finished
    rnd = random.Random(seed * 7 + P)
    pages = rnd.choice([24, 40, 400])
    pair = Pair(pages, P, rnd.sample(range(pages), pages))
    try:
        # some cache first (finished requests), so that appends may evict
        for _ in range(3):
            base = [rnd.randint(0, 2) for _ in range(rnd.randint(0, 9))]
            pair.batch([base + [rnd.randint(0, 2) for _ in range(rnd.randint(0, 6))] for _ in range(2)])
            while pair.live:
                pair.finish(0)
        base = [rnd.randint(0, 2) for _ in range(rnd.randint(0, 12))]
        seqs = []
        for _ in range(rnd.randint(1, 5)):
            if seqs and rnd.random() < 0.3:
                seqs.append(list(seqs[0]))     # an identical request: its context ends in a shared segment
            else:
                seqs.append(base[:rnd.randint(0, len(base))] + [rnd.randint(0, 2) for _ in range(rnd.randint(0, 5))])
        try:
            rows, lasts, _ = build_batch(pair.o, seqs)
        except NoSlotsError:
            return "no slots at build"
        B = len(seqs)
        ld = max(len(s) for s in seqs) + steps
        g = sgl.sgl_groups_create()
        out = sgl.sgl_build_batch(pair.t, seqs, ld=ld, groups=g)
        table, seq = out["req_to_token"], out["seq_lens"]
        toks = np.zeros((B, ld), dtype=np.int32)
        for r, s in enumerate(seqs):
            toks[r, :len(s)] = s
        # identical requests keep generating identical tokens half of the time
        same = rnd.random() < 0.5
        status = "ok"
        for step in range(steps):
            try:
                append_step(pair.o, rows)
                failed = False
            except NoSlotsError:
                failed = True
            if failed:
                with pytest.raises(sgl.SglError) as e:
                    sgl.sgl_batch_append(pair.t, table, seq, g)
                assert e.value.status == -2
                status = "no slots at step %d" % step
                pair.check_stats()
                break
            sgl.sgl_batch_append(pair.t, table, seq, g)
            new = [rnd.randint(0, 2) for _ in range(B)]
            for r in range(B):
                if same and seqs[r] == seqs[0] and toks[r, :seq[r] - 1].tolist() == toks[0, :seq[0] - 1].tolist():
                    new[r] = new[0]
                toks[r, seq[r] - 1] = new[r]
            for r, row in enumerate(rows):
                assert seq[r] == len(row)
                assert table[r, :len(row)].tolist() == list(row)
                assert np.all(table[r, len(row):] == -1)
            ogroups = prefix_groups(table, seq)
            _groups_eq(_lib_groups(g), ogroups)
            pair.check_stats()
        for r in range(B):
            cache_finished(pair.o, lasts[r], toks[r, :len(rows[r])].tolist(), rows[r])
        sgl.sgl_tree_cache_finished_batch(pair.t, toks, out)
        sgl.sgl_groups_destroy(g)
        pair.check_stats()
        assert sgl.sgl_tree_stats(pair.t)["locked_tokens"] == 0
        # the same cache: the same matches of every finished sequence, the same eviction
        for r in range(B):
            pair.match(toks[r, :len(rows[r])].tolist())
        pair.evict(rnd.randint(1, 4 * P))
        pair.alloc_free(rnd.randint(0, 3 * P))
        pair.check_stats()
        return status
    finally:
        pair.close()


@pytest.mark.parametrize("P", [1, 2, 4])
@pytest.mark.parametrize("seed", range(20))
def test_append_and_cache_finished_bit_exact(P, seed):
    _append_run(P, seed, steps=1 + seed % 9)


def test_append_runs_out_of_slots_like_the_oracle():
    """Small pools: some runs end with SGL_ERR_NO_SLOTS at an append, as the
    oracle does at the same step."""
    statuses = [_append_run(P, 100 + s, steps=60) for P in (1, 2) for s in range(12)]
    assert any(st.startswith("no slots at step") for st in statuses), statuses


def test_append_growing_batch_keeps_the_tree_small():
    """Decode steps through sgl_batch_append leave the tree alone: its node
    count after many steps equals the count after the build, and the groups
    still equal those computed from the table."""
    w = W.get("llama3_8b_decode_small")
    seqs = W.make_batch(w, 0).all_tokens()
    S = 1 << 15
    t = sgl.sgl_tree_create(S, 1, np.arange(S, dtype=np.int32))
    g = sgl.sgl_groups_create()
    steps = 40
    try:
        out = sgl.sgl_build_batch(t, seqs, ld=max(len(s) for s in seqs) + steps, groups=g)
        n0 = sgl.sgl_tree_stats(t)["num_nodes"]
        for _ in range(steps):
            sgl.sgl_batch_append(t, out["req_to_token"], out["seq_lens"], g)
        assert sgl.sgl_tree_stats(t)["num_nodes"] == n0
        _groups_eq(_lib_groups(g), prefix_groups(out["req_to_token"], out["seq_lens"]))
        g2 = sgl.sgl_groups_create()
        sgl.sgl_groups_from_table(out["req_to_token"], out["seq_lens"], g2)
        _groups_eq(_lib_groups(g), _lib_groups(g2))
        sgl.sgl_groups_destroy(g2)
    finally:
        sgl.sgl_groups_destroy(g)
        sgl.sgl_tree_destroy(t)


def test_append_and_cache_finished_refuse_bad_input():
    t = sgl.sgl_tree_create(64, 2, np.arange(32, dtype=np.int32))
    g = sgl.sgl_groups_create()
    try:
        seqs = [[1, 2, 3], [1, 2, 3, 4]]
        out = sgl.sgl_build_batch(t, seqs, ld=4, groups=g)
        before = sgl.sgl_tree_stats(t)
        tab, seq = out["req_to_token"], out["seq_lens"]
        with pytest.raises(sgl.SglError) as e:      # row 1 is already ld long
            sgl.sgl_batch_append(t, tab, seq, g)
        assert e.value.status == -1
        assert seq.tolist() == [3, 4] and sgl.sgl_tree_stats(t) == before
        empty = sgl.sgl_groups_create()
        tab2 = np.full((2, 8), -1, dtype=np.int32)
        tab2[:, :4] = tab
        with pytest.raises(sgl.SglError) as e:      # groups of another batch
            sgl.sgl_batch_append(t, tab2, seq, empty)
        assert e.value.status == -1
        sgl.sgl_groups_destroy(empty)
        bad = tab2.copy()
        bad[0, 2] = bad[0, 2] + 1                   # tail slot followed by another page's slot
        with pytest.raises(sgl.SglError) as e:
            sgl.sgl_batch_append(t, bad, seq.copy(), None)
        assert e.value.status == -1
        assert sgl.sgl_tree_stats(t) == before
        last = int(out["last_nodes"][1])
        with pytest.raises(sgl.SglError) as e:      # tokens disagree with the held path
            sgl.sgl_tree_cache_finished(t, last, [1, 9, 3, 4], tab[1], 4)
        assert e.value.status == -1
        with pytest.raises(sgl.SglError) as e:      # slots disagree with the held path
            sgl.sgl_tree_cache_finished(t, last, [1, 2, 3, 4], tab[0][[0, 1, 2, 2]] * 0 + 30, 4)
        assert e.value.status == -1
        assert sgl.sgl_tree_stats(t) == before
        assert sgl.sgl_tree_cache_finished(t, last, [1, 2, 3, 4], tab[1], 4) == 0
        with pytest.raises(sgl.SglError) as e:      # its reference is gone
            sgl.sgl_tree_cache_finished(t, last, [1, 2, 3, 4], tab[1], 4)
        assert e.value.status == -6
    finally:
        sgl.sgl_groups_destroy(g)
        sgl.sgl_tree_destroy(t)
