"""Oracle cache-aware scheduling simulation over the oracle trie.

Test infrastructure only (see ``oracle/__init__``).

Sources (page title, section):
  * "SGLang：从前端 DSL 到 SRT 服务运行时" (oripoin.cn/posts/sglang-runtime),
    section "用基数树实现前缀复用": cache-aware scheduling serves the waiting
    request with the longest shared (cached) prefix first, approximating a
    depth-first walk of the tree; leaf-first LRU eviction; reference counts
    keep running requests' nodes.
  * The CS349D lecture-16 notes (semidirectx.com), §3.1-3.3: a runtime with
    continuous batching (each request past prefill decodes one token per
    round), a per-round budget of prompt tokens (chunked prefill), FCFS or
    longest-prefix-first queueing in which a request whose uncached prefix
    largely coincides with one admitted in the same round waits for the next
    round, and insertion of the prompt into the tree when its prefill
    completes (inserting only at request end loses sharing between running
    requests).

Readings: rounds are discrete; a request is admitted
only if slots for its uncached prompt and its whole output can be allocated
(evicting LRU leaves), and the first allocation failure ends admission for
the round; the deferral rule compares the next min(defer_tokens, uncached)
prompt tokens of requests with equal cached lengths; a finished request
inserts its whole sequence, releases its references and frees its partial
tail page; a request that depends on another arrives ``delay`` rounds after
that one finishes.  Every step is taken in the order the C library's
``sgl_sim_run`` takes it, so both produce the same numbers.
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
