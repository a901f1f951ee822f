"""Cache-aware scheduling simulation: the C library (sgl_sim_run over the
native radix tree) against the oracle (oracle/sched.py over the oracle trie),
request by request, and the oracle against closed forms -- CPU only.

Pins for the oracle: token accounting identities; a lone request's rounds in
closed form; few-shot requests sharing an application prompt all hit it after
the first one (longest-prefix-first with deferral, insertion at prefill
completion, ample pool) but none hit it when every request runs at once and
prompts enter the tree only at request end (the interaction the lecture notes
describe); every turn of a conversation hits its whole history when the pool
is large enough; and two traces worked out by hand in their docstrings, which
fix hit counts, evictions and admission rounds from the pages' rules alone
(longest-prefix-first against FCFS in a pool that holds one branch, and the
deferral rule), held against both the oracle and the native simulator.
"""

import numpy as np
import pytest

import radixattention_prefix_shared_radix_gb300 as sgl
import workloads as W
from oracle.sched import AT_FINISH, AT_PREFILL, FCFS, LPM, simulate
from oracle.tree import RadixTrie


def _both(reqs, S, P, **cfg):
    order = np.random.default_rng([S, P]).permutation(S // P).astype(np.int32)
    t = sgl.sgl_tree_create(S, P, order)
    try:
        per, st = sgl.sgl_sim_run(t, reqs, **cfg)
        tree_after = sgl.sgl_tree_stats(t)
    finally:
        sgl.sgl_tree_destroy(t)
    trie = RadixTrie(S, P, order)
    per2, st2 = simulate(trie, reqs, **cfg)
    return per, st, per2, st2, tree_after, trie


@pytest.mark.parametrize("policy", [FCFS, LPM])
@pytest.mark.parametrize("insert_at", [AT_PREFILL, AT_FINISH])
@pytest.mark.parametrize("S,P", [(6000, 1), (1500, 1), (6000, 4), (1600, 4)])
def test_few_shot_native_equals_oracle(policy, insert_at, S, P):
    reqs = W.few_shot_trace(apps=3, sys_len=120, n_requests=24, question=(5, 30), output=(3, 12), spread=6)
    per, st, per2, st2, tree_after, trie = _both(reqs, S, P, policy=policy, insert_at=insert_at, prefill_budget=150,
                                                 max_running=6, defer_tokens=16)
    assert per == per2 and st == st2
    assert tree_after["tree_tokens"] == trie.tree_tokens()


@pytest.mark.parametrize("policy", [FCFS, LPM])
@pytest.mark.parametrize("S", [20000, 350])
def test_multi_turn_native_equals_oracle(policy, S):
    reqs = W.multi_turn_trace(conversations=6, turns=4, sys_len=50, user=(4, 20), output=(4, 20), delay=(1, 6))
    per, st, per2, st2, tree_after, trie = _both(reqs, S, 1, policy=policy, insert_at=AT_PREFILL,
                                                 prefill_budget=128, max_running=4, defer_tokens=8)
    assert per == per2 and st == st2
    assert st["evicted_tokens"] > 0 or S == 20000


def test_accounting_identities():
    reqs = W.few_shot_trace(apps=2, sys_len=40, n_requests=10, question=(3, 9), output=(2, 5))
    per, st = simulate(RadixTrie(4000, 1), reqs, policy=LPM, prefill_budget=50, max_running=3, defer_tokens=8)
    assert st["prompt_tokens"] == sum(len(r["prompt"]) for r in reqs)
    assert st["cached_tokens"] + st["prefill_tokens"] == st["prompt_tokens"]
    assert st["decode_tokens"] == sum(len(r["output"]) for r in reqs)
    assert st["cached_tokens"] == sum(p["cached_tokens"] for p in per)
    for p in per:
        assert p["arrive_round"] <= p["admit_round"] <= p["prefill_done_round"] < p["finish_round"] < st["rounds"]


@pytest.mark.parametrize("L,B,out", [(1, 1, 1), (100, 7, 5), (64, 64, 3), (65, 64, 1)])
def test_lone_request_rounds_closed_form(L, B, out):
    reqs = [dict(prompt=np.arange(1, L + 1), output=np.arange(1, out + 1), arrive_round=2)]
    per, st = simulate(RadixTrie(1000, 1), reqs, prefill_budget=B)
    done = 2 + (L + B - 1) // B - 1          # last prefill round
    assert per[0]["prefill_done_round"] == done
    assert per[0]["finish_round"] == done + out   # one token per round from the next round on
    assert st["rounds"] == done + out + 1


def test_few_shot_sharing_needs_insertion_at_prefill():
    apps, sys_len, n = 4, 64, 20
    reqs = W.few_shot_trace(apps=apps, sys_len=sys_len, n_requests=n, question=(5, 10), output=(4, 8))
    firsts = {}
    for i, r in enumerate(reqs):
        firsts.setdefault(tuple(r["prompt"][:sys_len]), i)
    # longest-prefix-first with deferral, prompts inserted at prefill completion
    per, st = simulate(RadixTrie(100000, 1), reqs, policy=LPM, insert_at=AT_PREFILL, prefill_budget=4096,
                       max_running=n, defer_tokens=16)
    for i, p in enumerate(per):
        assert p["cached_tokens"] == (0 if i in firsts.values() else sys_len)
    assert st["cached_tokens"] == (n - len(firsts)) * sys_len
    # everything admitted at once, prompts inserted only at request end: no sharing
    per, st = simulate(RadixTrie(100000, 1), reqs, policy=FCFS, insert_at=AT_FINISH, prefill_budget=4096,
                       max_running=n)
    assert st["cached_tokens"] == 0


def test_multi_turn_hits_whole_history_with_ample_pool():
    reqs = W.multi_turn_trace(conversations=3, turns=4, sys_len=30, user=(4, 9), output=(3, 7), delay=(1, 3))
    per, st = simulate(RadixTrie(100000, 1), reqs, policy=FCFS, prefill_budget=512, max_running=8)
    for i, r in enumerate(reqs):
        dep = r.get("depends_on", -1)
        if dep >= 0:
            hist = len(reqs[dep]["prompt"]) + len(reqs[dep]["output"])
            assert per[i]["cached_tokens"] == hist
        elif i > 0:
            assert per[i]["cached_tokens"] >= 0


def _two_system_prompt_trace():
    """Six requests, all arriving in round 0, alternating between two
    8-token system prompts X and Y; each has its own 4-token question and a
    1-token answer, so a whole sequence is 13 tokens."""
    X, Y = list(range(100, 108)), list(range(200, 208))
    return [dict(prompt=(X if i % 2 == 0 else Y) + [300 + 10 * i + k for k in range(4)], output=[900 + i],
                 arrive_round=0) for i in range(6)]


@pytest.mark.parametrize("native", [False, True])
def test_tight_pool_longest_prefix_first_by_hand(native):
    """Longest-prefix-first (an approximate depth-first walk of the tree,
    oripoin.cn "用基数树实现前缀复用") against FCFS when the KV pool holds
    only one request's branch (lecture-16 notes §3.3: with little KV room the
    ordering decides which prefix survives).  Pool 16 slots, page 1, one
    request running at a time, prefill in one round, insertion at prefill.

    Worked by hand (r_i = request i; X-requests are even):
      FCFS runs r0..r5 in order, one per two rounds (admit, then decode and
      finish).  r0 caches nothing and leaves X+q0+a0 (13) in the tree.  r1
      (Y) needs 13 slots with 3 free: the LRU leaf chain a0, q0, X[7..3] goes
      (10), leaving X[0..2].  r2 then matches only X[0..2] (3), needs 10 and
      evicts the Y branch down to Y[0..2]; every later request likewise finds
      3 tokens of its system prompt.  Cached: 0, 0, 3, 3, 3, 3 (12);
      evicted 10 per request after r0 (50); admitted in rounds 0, 2, ..., 10.
      Longest-prefix-first: after r0, the X-requests match 8 and go first
      (r2 in round 2, r4 in round 4), each evicting only the previous
      question's branch (r2: a0 and one token of q0, 2; r4: the rest of q0
      and a2 plus one token of q2, 5).  Then r1 (round 6) finds no Y and
      evicts all but X[0..2] (13); r3 and r5 then match Y fully (evicting 5
      each).  Cached: 0, 0, 8, 8, 8, 8 (32); evicted 30; admitted in rounds
      0, 6, 2, 8, 4, 10.
    The native simulator is held to the same numbers."""
    reqs = _two_system_prompt_trace()
    cfg = dict(insert_at=AT_PREFILL, prefill_budget=1000, max_running=1)
    expect = {FCFS: ([0, 0, 3, 3, 3, 3], [0, 2, 4, 6, 8, 10], 12, 50),
              LPM: ([0, 0, 8, 8, 8, 8], [0, 6, 2, 8, 4, 10], 32, 30)}
    for policy, (cached, admit, total, evicted) in expect.items():
        if native:
            t = sgl.sgl_tree_create(16, 1, np.arange(16, dtype=np.int32))
            try:
                per, st = sgl.sgl_sim_run(t, reqs, policy=policy, **cfg)
            finally:
                sgl.sgl_tree_destroy(t)
        else:
            per, st = simulate(RadixTrie(16, 1), reqs, policy=policy, **cfg)
        assert [p["cached_tokens"] for p in per] == cached
        assert [p["admit_round"] for p in per] == admit
        assert [p["finish_round"] for p in per] == [a + 1 for a in admit]
        assert st["cached_tokens"] == total and st["evicted_tokens"] == evicted and st["rounds"] == 12


@pytest.mark.parametrize("native", [False, True])
def test_deferral_by_hand(native):
    """The deferral rule (lecture-16 notes §3, queueing bullet): two requests
    with the same 8-token system prompt arrive together in round 0; room for
    both.  FCFS admits both at once, neither finds anything cached.
    Longest-prefix-first with deferral admits the first, defers the second
    (its first 4 uncached tokens equal those of a request admitted this
    round, with the same cached length 0), inserts the first prompt at its
    prefill in round 0, and admits the second in round 1 with all 8 system
    tokens cached."""
    X = list(range(100, 108))
    reqs = [dict(prompt=X + [300, 301], output=[900, 901], arrive_round=0),
            dict(prompt=X + [310, 311], output=[910, 911], arrive_round=0)]
    cfg = dict(insert_at=AT_PREFILL, prefill_budget=1000, max_running=4, defer_tokens=4)
    for policy, cached, admit in ((FCFS, [0, 0], [0, 0]), (LPM, [0, 8], [0, 1])):
        if native:
            t = sgl.sgl_tree_create(1000, 1, None)
            try:
                per, st = sgl.sgl_sim_run(t, reqs, policy=policy, **cfg)
            finally:
                sgl.sgl_tree_destroy(t)
        else:
            per, st = simulate(RadixTrie(1000, 1), reqs, policy=policy, **cfg)
        assert [p["cached_tokens"] for p in per] == cached
        assert [p["admit_round"] for p in per] == admit
