"""Oracle cache-aware scheduling simulation over the oracle trie.

Test infrastructure only (see ``oracle/__init__``).

What the pages fix, and where:
  * Queue order.  "SGLang：从前端 DSL 到 SRT 服务运行时" (oripoin.cn), section
    "用基数树实现前缀复用", fourth bullet: the cache-aware scheduler picks the
    waiting request whose shared (cached) prefix is longest, which walks the
    tree roughly depth first; the paper's Theorem 3.1 makes that order
    optimal for the hit rate when the cache holds at most one longest
    request.  The CS349D lecture-16 notes (semidirectx.com) §3, fourth bullet
    of the mini-runtime list: the policy is FCFS or longest-prefix-first.
  * Deferral.  Same bullet of the notes: under longest-prefix-first, a
    request whose not-yet-cached prefix largely coincides with a request
    admitted in the same round waits for the next round.
  * Rounds.  Notes §3, second and third bullets: continuous batching (every
    request whose prefill is done decodes one token per round) and chunked
    prefill (what is left of a per-round budget of prompt tokens goes to the
    requests still in prefill).
  * Insertion time.  Notes §3.1, "一个相互作用的例子": the prompt enters the
    tree when its prefill completes; inserting only at request end loses all
    sharing between requests that run at the same time.
  * Eviction and references.  oripoin.cn, same section, first two bullets:
    leaf-first LRU eviction, and nodes referenced by running requests are
    never evicted; the cache and the running requests share one pool (third
    bullet), so admission can evict.
  * Tight memory.  Notes §3.3: with little KV room the ordering changes which
    prefixes survive eviction.

Readings where the pages stop short (each is ours):
  1. A round runs, in this order: arrivals; queue ordering (match lengths
     from the trie, which refreshes the matched path's LRU stamps); admission
     in queue order while fewer than ``max_running`` requests run; prefill of
     up to ``prefill_budget`` prompt tokens in admission order; one decode
     token for every request whose prefill finished in an earlier round;
     finishing.
  2. Admission allocates the uncached prompt and the whole output at once
     (evicting LRU leaves as needed); the first allocation failure ends
     admission for the round.
  3. "Largely coincides" means: equal cached length and equal next
     ``min(defer_tokens, uncached length)`` prompt tokens.
  4. A finished request inserts its whole sequence, releases its reference
     and frees a partial tail page.
  5. A request that depends on another (the next turn of a conversation)
     arrives ``delay`` rounds after that one finishes.
"""

from oracle.tree import NoSlotsError

FCFS, LPM = 0, 1
AT_PREFILL, AT_FINISH = 0, 1


def simulate(trie, requests, policy=LPM, insert_at=AT_PREFILL, prefill_budget=2048, max_running=256,
             defer_tokens=0, max_rounds=1 << 30):
    """Run the trace; returns (per-request dicts, stats dict).

    requests: dicts with prompt, output (lists of token ids, non-empty) and
    arrive_round, or depends_on (an earlier index) and delay.
    """
    n = len(requests)
    R = []
    for i, q in enumerate(requests):
        dep = int(q.get("depends_on", -1))
        R.append(dict(prompt=[int(t) for t in q["prompt"]], seq=[int(t) for t in q["prompt"]] + [int(t) for t in q["output"]],
                      out_len=len(q["output"]), dep=dep, delay=int(q.get("delay", 0)),
                      arrive=int(q.get("arrive_round", 0)) if dep < 0 else -1,
                      queued=False, cached=0, remaining=0, generated=0, prefilled=False, prefill_round=-1,
                      lock=None, row=[]))
    per = [dict(arrive_round=-1, admit_round=-1, cached_tokens=0, prefill_done_round=-1, finish_round=-1)
           for _ in range(n)]
    stats = dict(rounds=0, prompt_tokens=0, cached_tokens=0, prefill_tokens=0, decode_tokens=0, evicted_tokens=0)
    waiting, running = [], []
    finished, rnd = 0, 0
    while finished < n:
        if rnd >= max_rounds:
            raise RuntimeError("max_rounds reached")
        # 1. arrivals in (arrival round, index) order
        arriving = sorted((i for i in range(n) if not R[i]["queued"] and 0 <= R[i]["arrive"] <= rnd),
                          key=lambda i: (R[i]["arrive"], i))
        for i in arriving:
            R[i]["queued"] = True
            per[i]["arrive_round"] = R[i]["arrive"]
            waiting.append(i)
        # 2. queue order: FCFS, or longest cached prefix first (stable)
        order = list(waiting)
        if policy == LPM:
            lens = {i: trie.match(R[i]["prompt"])[0] for i in order}
            order = sorted(order, key=lambda i: -lens[i])
        # 3. admission
        admitted_now = []
        for i in order:
            if len(running) >= max_running:
                break
            r = R[i]
            m, mslots, mnode = trie.match(r["prompt"])
            if policy == LPM and defer_tokens > 0:
                k = min(defer_tokens, len(r["prompt"]) - m)
                if k > 0 and any(R[j]["cached"] == m and len(R[j]["prompt"]) >= m + k and
                                 R[j]["prompt"][m:m + k] == r["prompt"][m:m + k] for j in admitted_now):
                    continue
            trie.lock(mnode)
            need = len(r["seq"]) - m
            before = trie.tree_tokens()
            try:
                fresh = trie.alloc(need)
            except NoSlotsError:
                stats["evicted_tokens"] += before - trie.tree_tokens()
                trie.unlock(mnode)
                break
            stats["evicted_tokens"] += before - trie.tree_tokens()
            r.update(lock=mnode, cached=m, remaining=len(r["prompt"]) - m, row=list(mslots) + list(fresh))
            per[i]["admit_round"] = rnd
            per[i]["cached_tokens"] = m
            stats["prompt_tokens"] += len(r["prompt"])
            stats["cached_tokens"] += m
            admitted_now.append(i)
            running.append(i)
            waiting.remove(i)
        # 4. prefill within the budget, in admission order
        budget = prefill_budget
        for i in running:
            r = R[i]
            if r["prefilled"] or budget == 0:
                continue
            t = min(r["remaining"], budget)
            r["remaining"] -= t
            budget -= t
            stats["prefill_tokens"] += t
            if r["remaining"] == 0:
                r["prefilled"] = True
                r["prefill_round"] = rnd
                per[i]["prefill_done_round"] = rnd
                if insert_at == AT_PREFILL:
                    _, last = trie.insert(r["prompt"], r["row"][:len(r["prompt"])])
                    trie.lock(last)
                    trie.unlock(r["lock"])
                    r["lock"] = last
        # 5. decode one token each; finish
        still = []
        for i in running:
            r = R[i]
            if r["prefilled"] and r["prefill_round"] < rnd:
                r["generated"] += 1
                stats["decode_tokens"] += 1
            if r["prefilled"] and r["generated"] == r["out_len"]:
                _, last = trie.insert(r["seq"], r["row"])
                trie.unlock(r["lock"])
                L = len(r["seq"])
                n_full = L // trie.P * trie.P
                if L > n_full:
                    trie.free_slots(r["row"][n_full:])
                per[i]["finish_round"] = rnd
                finished += 1
                for j in range(i + 1, n):
                    if R[j]["dep"] == i:
                        R[j]["arrive"] = rnd + R[j]["delay"]
            else:
                still.append(i)
        running = still
        rnd += 1
    stats["rounds"] = rnd
    return per, stats
