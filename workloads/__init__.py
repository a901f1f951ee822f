"""Seeded synthetic inputs for the RadixAttention hot path.

Shared by the oracle-side tests, the CUDA-side tests and ``bench.py``.  This
module only DRAWS inputs (token ids, lengths, the slot/page free-list
permutation, Q, K, V); it holds none of the method's arithmetic (no matching,
allocation, grouping or attention).

Workloads (shapes of the five configurations the hot path is measured on):
  1 tiny_fp32         4 requests sharing a 64-token prefix + 16-token
                      suffixes; Hq 4, Hkv 2, d 64, fp32, 1024-slot pool.
  2 llama3_8b_decode  64 requests sharing a 2048-token system prefix, each
                      with a uniform 64..512-token suffix; Hq 32, Hkv 8,
                      d 128, bf16, 2^20-slot pool.
  3 fork_tree         16 prompts x 1024 tokens, 8 forks each with a
                      256-token branch (128 requests); Llama-3-8B heads;
                      2^19-slot pool.
  4 extend            8 requests, each with its own cached 4096-token prefix
                      and 512 new tokens (causal); Hq 64, Hkv 8, d 128;
                      2^20-slot pool (the "1M-slot pool" of workload 2).
  5 multiturn         256 requests in groups of 4; per group one context
                      length L ~ lognormal(median 3000, sigma 1) capped to
                      [1, 32768]; the members share the first
                      16*floor(0.8*L/16) tokens; page size 16.
  5 multiturn_noshare the same lengths with no sharing.
  6 mla_decode        MLA (DeepSeek-Coder-V2-Lite attention shape after
                      weight absorption): 16 query heads over ONE stored
                      row per token of 576 elements (512-dim latent + 64-dim
                      position part), the output the first 512; the batch
                      of workload 2 (64 requests, 2048-token shared prefix,
                      64..512-token suffixes); bf16, 2^20-slot pool.
                      mla_decode_h128_small: 128 query heads (the
                      DeepSeek-V3 shape) at test size.
Scaled-down shapes of 2-5 (``*_small``) serve the element-by-element parity
tests; they keep every structural feature (sharing, forks, raggedness,
pages) at sizes the oracle finishes in seconds.

Seeds and draw order (seed = 1000 + workload number):
  * batch instance i:  default_rng([seed, 1, i]) draws lengths, then token
    ids segment by segment, then Q (float32 N(0,1)).
  * top-level first tokens: default_rng([seed, 2]).permutation(vocab); the
    top-level segments of instance i take consecutive entries, so distinct
    instances never share a tree path.
  * pool: default_rng([seed, 3]) draws the free-list permutation (of slots
    for page size 1, of pages otherwise); K and V are float32 N(0,1) drawn
    per fixed block of 2^22 elements from default_rng([seed, 3, 0|1, block]).
  * bf16 workloads round Q, K and V to bf16 (round-to-nearest-even, by
    torch on the host); both sides see the same bits.
Siblings (segments with the same parent) get distinct first tokens, so the
designed branch points are exactly where the sequences diverge.
"""

from dataclasses import dataclass, field
import math

import numpy as np

VOCAB = 32000
_POOL_BLOCK = 1 << 22


@dataclass(frozen=True)
class Workload:
    name: str
    number: int
    kind: str                 # "decode" or "extend"
    dtype: str                # "f32" or "bf16"
    Hq: int
    Hkv: int
    d: int
    page_size: int
    structure: tuple          # (builder name, parameters)
    num_slots: int = 0        # 0: sized from the structure (pool_factor x need)
    pool_factor: float = 1.25
    dv: int = 0               # MLA: output width (a prefix of the stored row); 0: not MLA

    @property
    def seed(self):
        return 1000 + self.number

    @property
    def G(self):
        return self.Hq // self.Hkv


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 1, "decode", "f32", 4, 2, 64, 1,
                          ("star", dict(n=4, prefix=64, suffix=(16, 16))), num_slots=1024),
    "llama3_8b_decode": Workload("llama3_8b_decode", 2, "decode", "bf16", 32, 8, 128, 1,
                                 ("star", dict(n=64, prefix=2048, suffix=(64, 512))), num_slots=1 << 20),
    "fork_tree": Workload("fork_tree", 3, "decode", "bf16", 32, 8, 128, 1,
                          ("fork", dict(prompts=16, prompt=(1024, 1024), forks=8, branch=(256, 256))),
                          num_slots=1 << 19),
    "extend": Workload("extend", 4, "extend", "bf16", 64, 8, 128, 1,
                       ("extend", dict(n=8, prefix=(4096, 4096), new=(512, 512))), num_slots=1 << 20),
    "multiturn": Workload("multiturn", 5, "decode", "bf16", 32, 8, 128, 16,
                          ("groups", dict(groups=64, size=4, median=3000, sigma=1.0, cap=32768, share=0.8))),
    "multiturn_noshare": Workload("multiturn_noshare", 5, "decode", "bf16", 32, 8, 128, 16,
                                  ("groups", dict(groups=64, size=4, median=3000, sigma=1.0, cap=32768, share=0.0))),
    "mla_decode": Workload("mla_decode", 6, "decode", "bf16", 16, 1, 576, 1,
                           ("star", dict(n=64, prefix=2048, suffix=(64, 512))), num_slots=1 << 20, dv=512),
    # scaled-down shapes for element-by-element parity
    "llama3_8b_decode_small": Workload("llama3_8b_decode_small", 2, "decode", "bf16", 32, 8, 128, 1,
                                       ("star", dict(n=8, prefix=300, suffix=(5, 130))), num_slots=8192),
    "fork_tree_small": Workload("fork_tree_small", 3, "decode", "bf16", 32, 8, 128, 1,
                                ("fork", dict(prompts=3, prompt=(90, 200), forks=4, branch=(1, 70))),
                                num_slots=4096),
    "extend_small": Workload("extend_small", 4, "extend", "bf16", 64, 8, 128, 1,
                             ("extend", dict(n=3, prefix=(0, 300), new=(1, 200))), num_slots=4096),
    "multiturn_small": Workload("multiturn_small", 5, "decode", "bf16", 32, 8, 128, 16,
                                ("groups", dict(groups=4, size=4, median=120, sigma=1.0, cap=700, share=0.8))),
    "mla_decode_small": Workload("mla_decode_small", 6, "decode", "bf16", 16, 1, 576, 1,
                                 ("star", dict(n=9, prefix=300, suffix=(5, 130))), num_slots=8192, dv=512),
    "mla_decode_h128_small": Workload("mla_decode_h128_small", 6, "decode", "bf16", 128, 1, 576, 1,
                                      ("star", dict(n=3, prefix=200, suffix=(1, 90))), num_slots=4096, dv=512),
}


def get(name):
    return WORKLOADS[name]


# --------------------------------------------------------------------------
# batch structure: a forest of segments; a request is a root-to-node chain
# --------------------------------------------------------------------------
@dataclass
class Batch:
    workload: Workload
    instance: int
    seg_parent: list = field(default_factory=list)   # parent segment id or -1
    seg_len: list = field(default_factory=list)
    seg_tokens: list = field(default_factory=list)   # np.int32 arrays
    req_chain: list = field(default_factory=list)    # list of segment-id lists
    cached_segments: int = 0                         # extend: chain[:k] is the cached prefix
    q: object = None                                 # float32 numpy (rounded later)

    def tokens(self, r):
        return np.concatenate([self.seg_tokens[s] for s in self.req_chain[r]]) if self.req_chain[r] else \
            np.zeros(0, dtype=np.int32)

    def all_tokens(self):
        return [self.tokens(r) for r in range(len(self.req_chain))]

    def cached_tokens(self, r):
        """Extend workloads: the tokens of request r that an earlier request cached."""
        chain = self.req_chain[r][:self.cached_segments]
        return np.concatenate([self.seg_tokens[s] for s in chain]) if chain else np.zeros(0, dtype=np.int32)

    def new_lens(self):
        return [sum(self.seg_len[s] for s in self.req_chain[r][self.cached_segments:])
                for r in range(len(self.req_chain))]


def _uniform_len(rng, lohi, n):
    lo, hi = lohi
    return [int(x) for x in rng.integers(lo, hi + 1, size=n)]


def _lengths(w, rng):
    """Draw the structure's lengths; returns (segments [(parent, len)], chains, cached)."""
    kind, p = w.structure
    segs, chains = [], []
    if kind == "star":
        suff = _uniform_len(rng, p["suffix"], p["n"])
        segs.append((-1, p["prefix"]))
        for r in range(p["n"]):
            segs.append((0, suff[r]))
            chains.append([0, r + 1])
        return segs, chains, 0
    if kind == "fork":
        plen = _uniform_len(rng, p["prompt"], p["prompts"])
        blen = _uniform_len(rng, p["branch"], p["prompts"] * p["forks"])
        for i in range(p["prompts"]):
            pid = len(segs)
            segs.append((-1, plen[i]))
            for f in range(p["forks"]):
                segs.append((pid, blen[i * p["forks"] + f]))
                chains.append([pid, len(segs) - 1])
        return segs, chains, 0
    if kind == "extend":
        pre = _uniform_len(rng, p["prefix"], p["n"])
        new = _uniform_len(rng, p["new"], p["n"])
        for r in range(p["n"]):
            if pre[r] > 0:
                segs.append((-1, pre[r]))
                segs.append((len(segs) - 1, new[r]))
                chains.append([len(segs) - 2, len(segs) - 1])
            else:
                segs.append((-1, new[r]))
                chains.append([len(segs) - 1])
        return segs, chains, 1
    if kind == "groups":
        z = rng.standard_normal(p["groups"])
        L = np.clip(np.rint(p["median"] * np.exp(p["sigma"] * z)), 1, p["cap"]).astype(np.int64)
        for g in range(p["groups"]):
            Lg = int(L[g])
            shared = 16 * int(math.floor(p["share"] * Lg / 16))
            if shared > 0:
                gid = len(segs)
                segs.append((-1, shared))
                for _ in range(p["size"]):
                    segs.append((gid, Lg - shared))
                    chains.append([gid, len(segs) - 1])
            else:
                for _ in range(p["size"]):
                    segs.append((-1, Lg))
                    chains.append([len(segs) - 1])
        return segs, chains, 0
    raise ValueError(kind)


def make_batch(name_or_workload, instance=0):
    """Token structure and Q of one batch instance."""
    w = get(name_or_workload) if isinstance(name_or_workload, str) else name_or_workload
    rng = np.random.default_rng([w.seed, 1, instance])
    segs, chains, cached = _lengths(w, rng)
    b = Batch(w, instance, cached_segments=cached)
    firsts = np.random.default_rng([w.seed, 2]).permutation(VOCAB)
    n_top = sum(1 for par, _ in segs if par < 0)
    top_iter = iter(firsts[instance * n_top:(instance + 1) * n_top])
    children = {}
    for sid, (par, n) in enumerate(segs):
        children.setdefault(par, []).append(sid)
    first_of = {}
    for par, kids in children.items():
        if par < 0:
            for sid in kids:
                first_of[sid] = int(next(top_iter))
        else:
            picks = rng.choice(VOCAB, size=len(kids), replace=False)
            for sid, t in zip(kids, picks):
                first_of[sid] = int(t)
    for sid, (par, n) in enumerate(segs):
        toks = rng.integers(0, VOCAB, size=n).astype(np.int32)
        if n > 0:
            toks[0] = first_of[sid]
        b.seg_parent.append(par)
        b.seg_len.append(n)
        b.seg_tokens.append(toks)
    b.req_chain = chains
    B = len(chains)
    if w.kind == "decode":
        b.q = rng.standard_normal((B, w.Hq, w.d), dtype=np.float32)
    else:
        N = sum(b.new_lens())
        b.q = rng.standard_normal((N, w.Hq, w.d), dtype=np.float32)
    return b


def make_new_kv(w, n_rows, instance=0):
    """K and V of n_rows new tokens [n_rows, Hkv, d] (float32 numpy, N(0,1)),
    for the KV write fused into extend: default_rng([seed, 4, instance])."""
    rng = np.random.default_rng([w.seed, 4, instance])
    k = rng.standard_normal((n_rows, w.Hkv, w.d), dtype=np.float32)
    v = rng.standard_normal((n_rows, w.Hkv, w.d), dtype=np.float32)
    return k, v


def make_queries(w, n_rows, instance=0):
    """Queries of n_rows tokens [n_rows, Hq, d] (float32 numpy, N(0,1)):
    default_rng([seed, 5, instance])."""
    return np.random.default_rng([w.seed, 5, instance]).standard_normal((n_rows, w.Hq, w.d), dtype=np.float32)


def pool_slots(w, instances=1):
    """Pool size in slots: fixed for most workloads; otherwise pool_factor x
    the pages the batch instances occupy (every segment rounded up to whole
    pages, plus one page per request for a partial tail)."""
    if w.num_slots:
        return w.num_slots
    P = w.page_size
    need = 0
    for i in range(instances):
        b = make_batch(w, i)
        need += sum(-(-n // P) for n in b.seg_len) + len(b.req_chain)
    return int(math.ceil(w.pool_factor * need)) * P


class RowView:
    """Float64 rows of a torch tensor pool: ``view[slots]`` -> numpy float64."""

    def __init__(self, tensor):
        self.t = tensor

    def __getitem__(self, slots):
        import torch
        idx = torch.from_numpy(np.asarray(slots, dtype=np.int64))
        return self.t.index_select(0, idx).double().numpy()


def make_pool(name_or_workload, num_slots=None, threads=None, only_k=False):
    """(free_order, K, V): the free-list permutation and the K/V pools.

    K and V are torch CPU tensors [S, Hkv, d] of the workload's dtype.  Each
    fixed block of 2^22 elements has its own generator
    default_rng([seed, 3, 0 for K / 1 for V, block]), so the values do not
    depend on how many threads fill them.
    """
    import os
    import torch
    from concurrent.futures import ThreadPoolExecutor
    w = get(name_or_workload) if isinstance(name_or_workload, str) else name_or_workload
    S = num_slots or pool_slots(w)
    order = np.random.default_rng([w.seed, 3]).permutation(S // w.page_size).astype(np.int32)
    tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    pools = []
    threads = threads or max(1, min(32, len(os.sched_getaffinity(0))))
    for which in range(1 if only_k else 2):
        t = torch.empty((S, w.Hkv, w.d), dtype=tdt)
        flat = t.view(-1)
        n = flat.numel()

        def fill(block, flat=flat, n=n, which=which):
            off = block * _POOL_BLOCK
            m = min(_POOL_BLOCK, n - off)
            x = np.random.default_rng([w.seed, 3, which, block]).standard_normal(m, dtype=np.float32)
            flat[off:off + m] = torch.from_numpy(x).to(tdt)

        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(-(-n // _POOL_BLOCK))))
        pools.append(t)
    return order, pools[0], (pools[1] if len(pools) > 1 else None)


def make_mla_pool(name_or_workload, num_slots=None):
    """(free_order, KV): the free-list permutation and the MLA pool, a torch
    CPU bf16 tensor [S, d] (one stored row per slot: latent then position
    part), drawn like make_pool's K pool."""
    w = get(name_or_workload) if isinstance(name_or_workload, str) else name_or_workload
    assert w.dv, "not an MLA workload"
    order, K, _ = make_pool(w, num_slots=num_slots, only_k=True)
    return order, K.view(K.shape[0], w.d)


def to_dtype(w, x):
    """Round a float32 numpy array to the workload's dtype as a torch CPU tensor."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x))
    return t if w.dtype == "f32" else t.to(torch.bfloat16)


# ---------------------------------------------------------------------------
# Request traces for the cache-aware scheduling simulation (seeded, synthetic)
# ---------------------------------------------------------------------------
def few_shot_trace(apps, sys_len, n_requests, question=(16, 64), output=(8, 32), seed=7, spread=0):
    """Few-shot serving: `apps` applications, each with its own system prompt
    of sys_len tokens; n_requests requests, each an application's system
    prompt followed by a fresh question, arriving at round 0 (or uniformly
    over `spread` rounds).  Tokens are ids in [1, VOCAB)."""
    rng = np.random.default_rng([seed, 6])
    sys = [rng.integers(1, VOCAB, size=sys_len).astype(np.int32) for _ in range(apps)]
    reqs = []
    for i in range(n_requests):
        app = int(rng.integers(0, apps))
        q = rng.integers(1, VOCAB, size=int(rng.integers(question[0], question[1] + 1))).astype(np.int32)
        out = rng.integers(1, VOCAB, size=int(rng.integers(output[0], output[1] + 1))).astype(np.int32)
        reqs.append(dict(prompt=np.concatenate([sys[app], q]), output=out,
                         arrive_round=int(rng.integers(0, spread + 1)) if spread else 0))
    return reqs


def multi_turn_trace(conversations, turns, sys_len, user=(16, 64), output=(16, 64), delay=(5, 20), seed=8):
    """Multi-turn chat: every conversation starts with a shared system prompt
    of sys_len tokens; turn t's prompt is turn t-1's prompt and output plus a
    new user message, arriving delay rounds after turn t-1 finishes (the first
    turns arrive over the first `conversations` rounds)."""
    rng = np.random.default_rng([seed, 7])
    sys = rng.integers(1, VOCAB, size=sys_len).astype(np.int32)
    reqs = []
    for c in range(conversations):
        hist = sys
        prev = -1
        for t in range(turns):
            u = rng.integers(1, VOCAB, size=int(rng.integers(user[0], user[1] + 1))).astype(np.int32)
            out = rng.integers(1, VOCAB, size=int(rng.integers(output[0], output[1] + 1))).astype(np.int32)
            prompt = np.concatenate([hist, u])
            r = dict(prompt=prompt, output=out)
            if prev < 0:
                r["arrive_round"] = c
            else:
                r["depends_on"], r["delay"] = prev, int(rng.integers(delay[0], delay[1] + 1))
            reqs.append(r)
            prev = len(reqs) - 1
            hist = np.concatenate([prompt, out])
    # requests must come after the ones they depend on: order by conversation turn
    return reqs


def quantize_e4m3(t, scale):
    """A pool for the FP8 KV cache: torch CPU tensor -> uint8 E4M3 codes of
    t / scale (torch's round-to-nearest conversion)."""
    import torch
    return (t.float() / float(scale)).to(torch.float8_e4m3fn).view(torch.uint8)
