"""Oracle prefix groups, defined directly from the slot table.

Test infrastructure only (see ``oracle/__init__``).

Source: bhfrc.com/news/45689 §1.3 (requests that share a path are branches
of one tree; the shared path is computed once) and §3.1 (each request only
remembers the node where it branches off); "SGLang：从前端 DSL 到 SRT 服务运行时"
section "用基数树实现前缀复用" (a shared prefix is computed once and referenced
many times).

Definition (reading; the pages give no data layout): position j of request r
belongs to the member set M(r, j) = { r' : seq_len[r'] > j and
req_to_token[r', 0..j] == req_to_token[r, 0..j] }.  A segment is a maximal run
of positions over which M stays the same; all members see the same run
[begin, end) and the same slots there.  Segments are listed once each, with
representative row = smallest member, ordered by (representative row, begin).
Because slots are unique to a tree path, equal slot prefixes are exactly the
shared tree path.
"""

import numpy as np


def prefix_groups_bruteforce(rows):
    """Direct transcription of the definition (pure Python; small inputs)."""
    B = len(rows)
    segs = {}
    for r in range(B):
        L = len(rows[r])
        prev = None
        start = 0
        for j in range(L + 1):
            if j < L:
                M = tuple(q for q in range(B)
                          if len(rows[q]) > j and list(rows[q][:j + 1]) == list(rows[r][:j + 1]))
            else:
                M = None
            if j > 0 and M != prev:
                segs[(prev, start)] = j
                start = j
            prev = M
    out = sorted(((min(M), b, e, M) for (M, b), e in segs.items()))
    return _pack(out)


def prefix_groups(req_to_token, seq_lens):
    """Same definition, vectorised per position with numpy (any size).

    ``req_to_token`` is an int array [B, ld]; ``seq_lens`` int [B].  The
    classes at position j refine the classes at j-1 by the slot at j; a class
    continues its parent's segment iff it kept all of the parent's members,
    otherwise the parent's segment ends at j.
    """
    table = np.asarray(req_to_token)
    lens = np.asarray(seq_lens, dtype=np.int64)
    B = len(lens)
    Lmax = int(lens.max()) if B else 0
    out = []
    prev_idx = prev_inv = prev_count = prev_begin = None
    label = np.zeros(B, dtype=np.int64)
    for j in range(Lmax):
        idx = np.nonzero(lens > j)[0]
        key = np.stack([label[idx], table[idx, j].astype(np.int64)], axis=1)
        uniq, inv, count = np.unique(key, axis=0, return_inverse=True, return_counts=True)
        inv = inv.reshape(-1)
        parent = uniq[:, 0]
        if j == 0:
            begin = np.zeros(len(uniq), dtype=np.int64)
        else:
            cont = count == prev_count[parent]
            begin = np.where(cont, prev_begin[parent], j)
            closed = np.setdiff1d(np.arange(len(prev_count)), parent[cont])
            for pc in closed:
                members = prev_idx[prev_inv == pc]
                out.append((int(members[0]), int(prev_begin[pc]), j, tuple(int(x) for x in members)))
        label = np.full(B, -1, dtype=np.int64)
        label[idx] = inv
        prev_idx, prev_inv, prev_count, prev_begin = idx, inv, count, begin
    if Lmax:
        for pc in range(len(prev_count)):
            members = prev_idx[prev_inv == pc]
            out.append((int(members[0]), int(prev_begin[pc]), Lmax, tuple(int(x) for x in members)))
    out.sort()
    return _pack(out)


def _pack(out):
    seg_row = np.array([o[0] for o in out], dtype=np.int32)
    seg_begin = np.array([o[1] for o in out], dtype=np.int32)
    seg_end = np.array([o[2] for o in out], dtype=np.int32)
    ptr = np.zeros(len(out) + 1, dtype=np.int32)
    members = []
    for i, o in enumerate(out):
        members.extend(o[3])
        ptr[i + 1] = len(members)
    return {
        "seg_begin": seg_begin,
        "seg_end": seg_end,
        "seg_row": seg_row,
        "seg_member_ptr": ptr,
        "seg_members": np.array(members, dtype=np.int32),
    }
