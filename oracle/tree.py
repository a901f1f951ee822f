"""Oracle radix cache: a plain per-page trie (per-token trie when page_size == 1).

Test infrastructure only (see ``oracle/__init__``).

Sources (page title, section):
  * "SGLang 深度拆解" (chenxutan.com/d/5669.html) §2.3: every node holds a
    token range, KV pointers, a reference count and an LRU timestamp; the
    match walks from the root one token at a time and stops at the first
    token with no child.
  * bhfrc.com/news/45689 §3.1: longest-prefix match on the radix tree, cost
    proportional to the matched length.  §3.2: a request adds one to the
    reference count of every node on its path and, when it ends, subtracts
    one from its last node back to the root; only nodes whose count is zero
    may be freed.
  * "SGLang：从前端 DSL 到 SRT 服务运行时" (oripoin.cn/posts/sglang-runtime),
    section "用基数树实现前缀复用": nodes hold contiguous token runs paged by
    one token or by multi-token pages; eviction is leaf-first LRU; reference
    counts protect in-flight requests; cache and running requests share one
    memory pool.
  * "SGLang 深度解读" (luoboask.github.io/fde-learning/opensource/sglang/),
    section "1. RadixCache": per-token trie with ``children[token]``,
    ``prefix_match`` returning (matched length, last node), and ``insert``.

Readings taken where the pages are silent:
  * Structure: one trie node per PAGE (a tuple of ``page_size`` token ids);
    for page_size == 1 this is the pages' per-token trie.  Matching and
    sharing happen in whole pages; a partially filled tail page is never
    inserted (it stays private to its request).
  * Reference counts follow the per-request lock/unlock of bhfrc §3.2 and
    oripoin, not the count-on-insert of the walkthrough page.
  * Insert of a path that already exists keeps the existing pages; a
    caller page that differs from the existing one at the same position is a
    duplicate and goes back to the free list.
  * Allocator: the free list starts as the given permutation of pages;
    ``alloc`` pops from the front, frees append to the back in the order they
    happen.
  * Clock: a logical counter, incremented once per ``match`` and once per
    ``insert`` call, stamped on every node of the path that call touches.
  * Eviction: repeatedly remove the unreferenced leaf with the smallest
    (last_access, creation id) until enough tokens are freed or none is left.
"""

from collections import deque


class NoSlotsError(RuntimeError):
    """The pool cannot supply the requested slots even after eviction."""


class StateError(RuntimeError):
    """A lock/unlock would drive a reference count below zero."""


class _Node:
    __slots__ = ("children", "parent", "key", "page", "ref", "last_access", "nid")

    def __init__(self, parent, key, page, nid):
        self.children = {}
        self.parent = parent
        self.key = key          # tuple of page_size token ids (None for root)
        self.page = page        # page id in the pool (None for root)
        self.ref = 0
        self.last_access = 0
        self.nid = nid          # creation order, the LRU tie-break


class RadixTrie:
    """Per-page trie over a slot pool of ``num_slots`` = pages * page_size."""

    def __init__(self, num_slots, page_size=1, free_order=None):
        if page_size < 1 or num_slots < 0 or num_slots % page_size:
            raise ValueError("num_slots must be a non-negative multiple of page_size")
        self.P = int(page_size)
        self.num_pages = num_slots // self.P
        if free_order is None:
            order = list(range(self.num_pages))
        else:
            order = [int(x) for x in free_order]
            if sorted(order) != list(range(self.num_pages)):
                raise ValueError("free_order must be a permutation of the pages")
        self.free = deque(order)
        self.clock = 0
        self._next_id = 1
        self.root = _Node(None, None, None, 0)

    # ------------------------------------------------------------------ util
    def _pages_of(self, tokens):
        n = len(tokens) // self.P
        return [tuple(int(t) for t in tokens[i * self.P:(i + 1) * self.P]) for i in range(n)]

    def _slots_of_page(self, page):
        return [page * self.P + o for o in range(self.P)]

    def _path_to_root(self, node):
        while node is not self.root:
            yield node
            node = node.parent

    def tree_tokens(self):
        """Number of tokens held by the trie (pages * page_size)."""
        count, stack = 0, [self.root]
        while stack:
            n = stack.pop()
            for c in n.children.values():
                count += self.P
                stack.append(c)
        return count

    def nodes(self):
        out, stack = [], [self.root]
        while stack:
            n = stack.pop()
            for c in n.children.values():
                out.append(c)
                stack.append(c)
        return out

    # ----------------------------------------------------------------- match
    def match(self, tokens):
        """Longest prefix of ``tokens`` present, in whole pages.

        Returns (matched_len, slots of the matched path, last node).  Stamps
        the matched path with a new clock value.
        """
        self.clock += 1
        node, slots = self.root, []
        for key in self._pages_of(tokens):
            child = node.children.get(key)
            if child is None:
                break
            node = child
            node.last_access = self.clock
            slots.extend(self._slots_of_page(node.page))
        return len(slots), slots, node

    # ---------------------------------------------------------------- insert
    def insert(self, tokens, slots):
        """Insert the full pages of ``tokens`` with their ``slots``.

        Returns (dup_len, last node).  ``dup_len`` counts tokens whose caller
        page was a duplicate of an existing page and was freed.
        """
        n_full = (len(tokens) // self.P) * self.P
        if len(slots) < n_full:
            raise ValueError("need a slot for every inserted token")
        keys = self._pages_of(tokens)
        pages = []
        for i in range(len(keys)):
            first = int(slots[i * self.P])
            if first % self.P:
                raise ValueError("slots of a page must start on a page boundary")
            page = first // self.P
            if [int(s) for s in slots[i * self.P:(i + 1) * self.P]] != self._slots_of_page(page):
                raise ValueError("slots of a page must be that page's consecutive slots")
            if not 0 <= page < self.num_pages:
                raise ValueError("slot out of range")
            pages.append(page)
        self.clock += 1
        node, dup = self.root, 0
        for key, page in zip(keys, pages):
            child = node.children.get(key)
            if child is None:
                child = _Node(node, key, page, self._next_id)
                self._next_id += 1
                node.children[key] = child
            elif child.page != page:
                dup += self.P
                self.free.append(page)
            node = child
            node.last_access = self.clock
        return dup, node

    # ------------------------------------------------------------ lock/unlock
    def lock(self, node):
        for n in self._path_to_root(node):
            n.ref += 1

    def unlock(self, node):
        path = list(self._path_to_root(node))
        if any(n.ref <= 0 for n in path):
            raise StateError("unlock below zero")
        for n in path:
            n.ref -= 1

    # ----------------------------------------------------------------- evict
    def _candidates(self):
        return [n for n in self.nodes() if not n.children and n.ref == 0]

    def evict(self, num_tokens):
        """Free at least ``num_tokens`` tokens by removing LRU leaves.

        Returns the number of tokens freed (may be less when every remaining
        leaf is referenced).
        """
        freed = 0
        while freed < num_tokens:
            cands = self._candidates()
            if not cands:
                break
            victim = min(cands, key=lambda n: (n.last_access, n.nid))
            del victim.parent.children[victim.key]
            self.free.append(victim.page)
            freed += self.P
        return freed

    # ----------------------------------------------------------------- alloc
    def alloc(self, num_tokens):
        """Slots for ``num_tokens`` tokens, in whole pages popped from the free list."""
        need = -(-int(num_tokens) // self.P)
        if len(self.free) < need:
            self.evict((need - len(self.free)) * self.P)
        if len(self.free) < need:
            raise NoSlotsError("pool exhausted")
        out = []
        for _ in range(need):
            out.extend(self._slots_of_page(self.free.popleft()))
        return out[:num_tokens]

    def free_slots(self, slots):
        """Return the pages holding ``slots`` to the free list (first-seen order)."""
        seen = []
        for s in slots:
            p = int(s) // self.P
            if p not in seen:
                seen.append(p)
        self.free.extend(seen)


def build_batch(trie, batch_tokens):
    """Assemble one batch: match, allocate the tail, insert, lock.

    For each request r in order: longest-prefix match; lock the matched node
    so allocation cannot evict it; allocate slots for the unmatched tail;
    row r of the table = matched slots ++ new slots; insert the full pages;
    lock the new last node and release the temporary lock.  The slots of a
    partial tail page (page_size > 1) stay private to the request.

    Source: the scheduler flow of "SGLang 深度解读" sections "2. Scheduler"
    and "5. Attention 层" (prefix match, then req_to_token rows of the
    matched prefix followed by newly allocated locations) and the per-request
    locking of bhfrc.com/news/45689 §3.2.

    Returns (rows, last_nodes, private_slots) where rows[r] is a list of
    slots of length len(batch_tokens[r]).  On NoSlotsError every lock taken
    by this call is released and the private tail pages it allocated are
    freed (in request order) before the error propagates; inserted nodes stay
    in the trie as unreferenced cache.
    """
    rows, lasts, private = [], [], []
    try:
        for toks in batch_tokens:
            L = len(toks)
            m, mslots, mnode = trie.match(toks)
            trie.lock(mnode)
            try:
                new = trie.alloc(L - m)
            except NoSlotsError:
                trie.unlock(mnode)
                raise
            row = list(mslots) + list(new)
            _, last = trie.insert(toks, row)
            trie.lock(last)
            trie.unlock(mnode)
            n_full = (L // trie.P) * trie.P
            rows.append(row)
            lasts.append(last)
            private.append(row[n_full:])
    except NoSlotsError:
        for node in lasts:
            trie.unlock(node)
        for tail in private:
            trie.free_slots(tail)
        raise
    return rows, lasts, private


def append_step(trie, rows):
    """One decode step of a running batch: every row gains one slot.

    The new tokens are not inserted into the trie: a sequence is cached when
    its request ends ("SGLang 深度拆解" (chenxutan.com) §1.3, the CPU
    scheduler's first step; the CS349D lecture-16 notes §3.1 insert the
    prompt at prefill completion and let the running request hold the
    rest).  Reading: "SGLang 深度解读" section "2. Scheduler" also shows a
    per-token insert of each decoded token; that variant is a sgl_build_batch
    of the grown sequences each step.  A row whose length is a multiple of
    the page size opens a fresh page (its first slot); any other row takes
    the next slot of its own partial tail page.

    Reading (the pages are silent on the order): the step's fresh pages come
    from one allocation of (rows needing a page) x page_size tokens and are
    handed to the rows in order.  ``rows`` (lists of slots) are extended in
    place.
    """
    need = sum(1 for row in rows if len(row) % trie.P == 0)
    fresh = trie.alloc(need * trie.P)
    k = 0
    for row in rows:
        if len(row) % trie.P == 0:
            row.append(fresh[k * trie.P])
            k += 1
        else:
            row.append(row[-1] + 1)


def cache_finished(trie, last, tokens, row):
    """A request ends: insert its whole sequence (full pages) with its slots,
    release the reference it held on ``last``, free its partial tail page.

    Source: a finished request's sequence and KV pages are inserted into the
    cache as the decode batch drops it ("SGLang 深度拆解" (chenxutan.com)
    §1.3; "SGLang 深度解读" section "2. Scheduler"); references released
    at request end (bhfrc.com/news/45689 §3.2).  Returns the duplicate
    tokens the insert freed.
    """
    dup, _ = trie.insert(tokens, row)
    trie.unlock(last)
    n_full = (len(row) // trie.P) * trie.P
    trie.free_slots(row[n_full:])
    return dup
