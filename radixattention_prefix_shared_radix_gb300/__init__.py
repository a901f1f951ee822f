"""GB300 RadixAttention hot path: Python binding of libsglattn.so.

Thin argument marshalling over the C ABI declared in ``include/sglattn.h``;
every step of the hot path runs in the native library (host radix tree and
planner in C++, attention in CUDA kernels for sm_103a).  Functions keep the C
names.  Device arguments are torch CUDA tensors (used only for their memory
and the current stream); host arguments are numpy arrays or Python lists.
There is no fallback: if the library is missing, every call raises.
"""

import ctypes
import os

import numpy as np

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = _build.LIB

SGL_OK = 0
SGL_DTYPE_F32 = 0
SGL_DTYPE_BF16 = 1
SGL_DTYPE_BF16_FP8KV = 2


class SglError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (%d)" % (where, _lib().sgl_status_string(status).decode(), status))


class SglTreeStats(ctypes.Structure):
    _fields_ = [("free_pages", ctypes.c_int64), ("tree_tokens", ctypes.c_int64),
                ("locked_tokens", ctypes.c_int64), ("evictable_tokens", ctypes.c_int64),
                ("num_nodes", ctypes.c_int64), ("clock", ctypes.c_int64)]


class SglPrefixGroups(ctypes.Structure):
    _fields_ = [("num_segments", ctypes.c_int32), ("num_members", ctypes.c_int32),
                ("seg_begin", ctypes.POINTER(ctypes.c_int32)), ("seg_end", ctypes.POINTER(ctypes.c_int32)),
                ("seg_row", ctypes.POINTER(ctypes.c_int32)), ("seg_member_ptr", ctypes.POINTER(ctypes.c_int32)),
                ("seg_members", ctypes.POINTER(ctypes.c_int32))]


class SglPlanInfo(ctypes.Structure):
    _fields_ = [("num_items", ctypes.c_int32), ("num_wide_items", ctypes.c_int32), ("num_partial_rows", ctypes.c_int32),
                ("num_merge_entries", ctypes.c_int32), ("chunk_tokens", ctypes.c_int32),
                ("upload_bytes", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64)]


class SglMlaParams(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_qo_heads", ctypes.c_int32), ("latent_dim", ctypes.c_int32),
                ("rope_dim", ctypes.c_int32), ("num_slots", ctypes.c_int64), ("page_size", ctypes.c_int32),
                ("sm_scale", ctypes.c_float), ("num_sms", ctypes.c_int32)]


class SglAttnParams(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("batch", ctypes.c_int32), ("num_qo_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_slots", ctypes.c_int64), ("sm_scale", ctypes.c_float), ("num_sms", ctypes.c_int32),
                ("host_prefix_lens", ctypes.POINTER(ctypes.c_int32)),
                ("host_extend_lens", ctypes.POINTER(ctypes.c_int32)),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


class SglSimConfig(ctypes.Structure):
    _fields_ = [("policy", ctypes.c_int32), ("insert_at", ctypes.c_int32), ("prefill_budget", ctypes.c_int64),
                ("max_running", ctypes.c_int32), ("defer_tokens", ctypes.c_int32), ("max_rounds", ctypes.c_int64)]


class SglSimRequest(ctypes.Structure):
    _fields_ = [("prompt", ctypes.POINTER(ctypes.c_int32)), ("prompt_len", ctypes.c_int64),
                ("output", ctypes.POINTER(ctypes.c_int32)), ("output_len", ctypes.c_int64),
                ("arrive_round", ctypes.c_int64), ("depends_on", ctypes.c_int32), ("delay", ctypes.c_int64)]


class SglSimResult(ctypes.Structure):
    _fields_ = [("arrive_round", ctypes.c_int64), ("admit_round", ctypes.c_int64), ("cached_tokens", ctypes.c_int64),
                ("prefill_done_round", ctypes.c_int64), ("finish_round", ctypes.c_int64)]


class SglSimStats(ctypes.Structure):
    _fields_ = [("rounds", ctypes.c_int64), ("prompt_tokens", ctypes.c_int64), ("cached_tokens", ctypes.c_int64),
                ("prefill_tokens", ctypes.c_int64), ("decode_tokens", ctypes.c_int64),
                ("evicted_tokens", ctypes.c_int64)]


SGL_SCHED_FCFS, SGL_SCHED_LPM = 0, 1
SGL_INSERT_AT_PREFILL, SGL_INSERT_AT_FINISH = 0, 1

_P = ctypes.c_void_p
_I32P = ctypes.POINTER(ctypes.c_int32)
_I64P = ctypes.POINTER(ctypes.c_int64)

_SIGS = {
    "sgl_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "sgl_last_cuda_error": (ctypes.c_int, []),
    "sgl_version": (ctypes.c_char_p, []),
    "sgl_tree_create": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int32, _I32P, ctypes.POINTER(_P)]),
    "sgl_tree_destroy": (None, [_P]),
    "sgl_tree_match": (ctypes.c_int, [_P, _I32P, ctypes.c_int64, _I64P, _I32P, _I64P]),
    "sgl_tree_insert": (ctypes.c_int, [_P, _I32P, _I32P, ctypes.c_int64, _I64P, _I64P]),
    "sgl_tree_lock": (ctypes.c_int, [_P, ctypes.c_int64]),
    "sgl_tree_unlock": (ctypes.c_int, [_P, ctypes.c_int64]),
    "sgl_tree_alloc": (ctypes.c_int, [_P, ctypes.c_int64, _I32P]),
    "sgl_tree_free": (ctypes.c_int, [_P, _I32P, ctypes.c_int64]),
    "sgl_tree_evict": (ctypes.c_int, [_P, ctypes.c_int64, _I64P]),
    "sgl_tree_stats": (ctypes.c_int, [_P, ctypes.POINTER(SglTreeStats)]),
    "sgl_build_batch": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.POINTER(_I32P), _I64P, _I32P, ctypes.c_int64,
                                       _I32P, _I32P, _I64P, _P]),
    "sgl_tree_finish": (ctypes.c_int, [_P, ctypes.c_int64, _I32P, ctypes.c_int64]),
    "sgl_tree_finish_batch": (ctypes.c_int, [_P, ctypes.c_int32, _I64P, _I32P, ctypes.c_int64, _I32P]),
    "sgl_batch_append": (ctypes.c_int, [_P, ctypes.c_int32, _I32P, ctypes.c_int64, _I32P, _P]),
    "sgl_tree_cache_finished": (ctypes.c_int, [_P, ctypes.c_int64, _I32P, _I32P, ctypes.c_int64, _I64P]),
    "sgl_tree_cache_finished_batch": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.POINTER(_I32P), _I64P, _I32P,
                                                     ctypes.c_int64, _I32P]),
    "sgl_groups_create": (ctypes.c_int, [ctypes.POINTER(_P)]),
    "sgl_groups_destroy": (None, [_P]),
    "sgl_groups_view": (ctypes.c_int, [_P, ctypes.POINTER(SglPrefixGroups)]),
    "sgl_groups_from_table": (ctypes.c_int, [_I32P, ctypes.c_int64, _I32P, ctypes.c_int32, _P]),
    "sgl_decode_plan": (ctypes.c_int, [ctypes.POINTER(SglAttnParams), _I32P, ctypes.POINTER(SglPrefixGroups),
                                       ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_size_t)]),
    "sgl_plan_destroy": (None, [_P]),
    "sgl_plan_info": (ctypes.c_int, [_P, ctypes.POINTER(SglPlanInfo)]),
    "sgl_plan_upload": (ctypes.c_int, [_P, _P, ctypes.c_size_t, _P]),
    "sgl_decode_attn": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_int64, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "sgl_decode_step": (ctypes.c_int, [_P, _P, ctypes.c_size_t, _P, _P, _P, _P, ctypes.c_int64, _P, _P, _P, _P, _P,
                                       _P, ctypes.c_size_t, _P, ctypes.c_size_t, _P]),
    "sgl_extend_workspace_bytes": (ctypes.c_int, [ctypes.POINTER(SglAttnParams), ctypes.POINTER(ctypes.c_size_t)]),
    "sgl_extend_attn": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_int64, _P, _P, ctypes.POINTER(SglAttnParams),
                                       _P, _P, _P, ctypes.c_size_t, _P]),
    "sgl_extend_attn_kvwrite": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, ctypes.c_int64, _P, _P,
                                               ctypes.POINTER(SglAttnParams), _P, _P, _P, ctypes.c_size_t, _P]),
    "sgl_check": (ctypes.c_int, [_P, _P]),
    "sgl_sim_run": (ctypes.c_int, [_P, ctypes.POINTER(SglSimConfig), ctypes.c_int32, ctypes.POINTER(SglSimRequest),
                                   ctypes.POINTER(SglSimResult), ctypes.POINTER(SglSimStats)]),
    "sgl_decode_attn_noalloc": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_int64, _P, _P, _P, _P, _P]),
    "sgl_mla_decode_plan": (ctypes.c_int, [ctypes.POINTER(SglMlaParams), _I32P, ctypes.POINTER(SglPrefixGroups),
                                           ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_size_t)]),
    "sgl_mla_decode_attn": (ctypes.c_int, [_P, _P, _P, ctypes.c_int64, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
}

_LIB = None


def _lib():
    """Load libsglattn.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libsglattn.so is not built (run __graft_entry__.build()); "
                               "there is no fallback path")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def exported_symbols():
    return list(_SIGS)


def _ok(st, where):
    if st != SGL_OK:
        raise SglError(st, where)


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr32(a):
    return a.ctypes.data_as(_I32P)


def _dev(t, what):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % what)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


# ------------------------------------------------------------------ tree
def sgl_version():
    return _lib().sgl_version().decode()


def sgl_status_string(status):
    return _lib().sgl_status_string(status).decode()


def sgl_tree_create(num_slots, page_size=1, free_order=None):
    h = _P()
    fo = None if free_order is None else _i32(free_order)
    _ok(_lib().sgl_tree_create(num_slots, page_size, None if fo is None else _ptr32(fo), ctypes.byref(h)),
        "sgl_tree_create")
    return h


def sgl_tree_destroy(tree):
    _lib().sgl_tree_destroy(tree)


def sgl_tree_match(tree, tokens):
    t = _i32(tokens)
    m, last = ctypes.c_int64(), ctypes.c_int64()
    slots = np.zeros(max(len(t), 1), dtype=np.int32)
    _ok(_lib().sgl_tree_match(tree, _ptr32(t), len(t), ctypes.byref(m), _ptr32(slots), ctypes.byref(last)),
        "sgl_tree_match")
    return m.value, slots[:m.value].copy(), last.value


def sgl_tree_insert(tree, tokens, slots):
    t, s = _i32(tokens), _i32(slots)
    dup, last = ctypes.c_int64(), ctypes.c_int64()
    _ok(_lib().sgl_tree_insert(tree, _ptr32(t), _ptr32(s), len(t), ctypes.byref(dup), ctypes.byref(last)),
        "sgl_tree_insert")
    return dup.value, last.value


def sgl_tree_lock(tree, node):
    _ok(_lib().sgl_tree_lock(tree, node), "sgl_tree_lock")


def sgl_tree_unlock(tree, node):
    _ok(_lib().sgl_tree_unlock(tree, node), "sgl_tree_unlock")


def sgl_tree_alloc(tree, n):
    out = np.zeros(max(n, 1), dtype=np.int32)
    _ok(_lib().sgl_tree_alloc(tree, n, _ptr32(out)), "sgl_tree_alloc")
    return out[:n].copy()


def sgl_tree_free(tree, slots):
    s = _i32(slots)
    _ok(_lib().sgl_tree_free(tree, _ptr32(s), len(s)), "sgl_tree_free")


def sgl_tree_evict(tree, num_tokens):
    f = ctypes.c_int64()
    _ok(_lib().sgl_tree_evict(tree, num_tokens, ctypes.byref(f)), "sgl_tree_evict")
    return f.value


def sgl_tree_stats(tree):
    s = SglTreeStats()
    _ok(_lib().sgl_tree_stats(tree, ctypes.byref(s)), "sgl_tree_stats")
    return {k: getattr(s, k) for k, _ in SglTreeStats._fields_}


def sgl_sim_run(tree, requests, policy=SGL_SCHED_LPM, insert_at=SGL_INSERT_AT_PREFILL, prefill_budget=2048,
                max_running=256, defer_tokens=0, max_rounds=1 << 30):
    """Cache-aware scheduling simulation (see sgl_sim_run in the C header).

    requests: list of dicts with prompt, output (int sequences), and either
    arrive_round or depends_on + delay.  Returns (per-request list of dicts,
    stats dict).
    """
    n = len(requests)
    keep = []
    arr = (SglSimRequest * max(1, n))()
    for i, r in enumerate(requests):
        pr, out = _i32(r["prompt"]), _i32(r["output"])
        keep += [pr, out]
        arr[i].prompt, arr[i].prompt_len = _ptr32(pr), len(pr)
        arr[i].output, arr[i].output_len = _ptr32(out), len(out)
        arr[i].arrive_round = int(r.get("arrive_round", 0))
        arr[i].depends_on = int(r.get("depends_on", -1))
        arr[i].delay = int(r.get("delay", 0))
    cfg = SglSimConfig(policy, insert_at, prefill_budget, max_running, defer_tokens, max_rounds)
    res = (SglSimResult * max(1, n))()
    st = SglSimStats()
    _ok(_lib().sgl_sim_run(tree, ctypes.byref(cfg), n, arr, res, ctypes.byref(st)), "sgl_sim_run")
    per = [{k: getattr(res[i], k) for k, _ in SglSimResult._fields_} for i in range(n)]
    return per, {k: getattr(st, k) for k, _ in SglSimStats._fields_}


def _out_i32(a, shape, name):
    """A caller's output array (int32, C-contiguous, of `shape`), or a new one."""
    if a is None:
        return np.empty(shape, dtype=np.int32)
    if not (isinstance(a, np.ndarray) and a.dtype == np.int32 and a.flags.c_contiguous and a.flags.writeable
            and a.shape == tuple(shape)):
        raise ValueError("%s must be a writeable C-contiguous int32 array of shape %s" % (name, tuple(shape)))
    return a


def sgl_build_batch(tree, token_lists, ld=None, groups=None, req_to_token=None, seq_lens=None, lens=None):
    """Returns dict(req_to_token [B, ld] int32, seq_lens, prefix_lens, last_nodes) (numpy).

    `token_lists` is a sequence of 1-D token arrays, or a [B, cap] int32
    C-contiguous matrix whose row r holds request r's `lens[r]` tokens
    first (a serving loop can append each step's token in place and pass
    the matrix with no per-step copy).

    `req_to_token` ([B, ld] int32, C-contiguous) and `seq_lens` ([B] int32)
    may be given to be written in place (e.g. pinned staging buffers that are
    copied to the device next); they are the arrays returned."""
    mat = isinstance(token_lists, np.ndarray) and token_lists.ndim == 2
    if mat:
        if token_lists.dtype != np.int32 or not token_lists.flags.c_contiguous:
            raise ValueError("a token matrix must be C-contiguous int32")
        B, cap = token_lists.shape
        lens = np.full(B, cap, dtype=np.int64) if lens is None else np.asarray(lens, dtype=np.int64).copy()
        if lens.shape != (B,) or (B and (lens.min() < 0 or lens.max() > cap)):
            raise ValueError("lens must give B lengths in [0, cap]")
    else:
        if lens is not None:
            raise ValueError("lens is given with a token matrix only")
        toks = [t if (isinstance(t, np.ndarray) and t.dtype == np.int32 and t.ndim == 1 and t.flags.c_contiguous)
                else _i32(t) for t in token_lists]
        B = len(toks)
        lens = np.fromiter((t.shape[0] for t in toks), dtype=np.int64, count=B)
    if req_to_token is not None:
        if ld is not None and int(ld) != req_to_token.shape[-1]:
            raise ValueError("ld disagrees with req_to_token")
        ld = req_to_token.shape[-1]
    ld = int(ld if ld is not None else max(1, int(lens.max()) if B else 1))
    table = _out_i32(req_to_token, (B, ld), "req_to_token")   # every entry is written (-1 past a row's length)
    seq = _out_i32(seq_lens, (B,), "seq_lens")
    pre = np.zeros(B, dtype=np.int32)
    last = np.zeros(B, dtype=np.int64)
    # the rows back to back in one array and their addresses computed in
    # one step (per-row ctypes or array-interface lookups cost more than
    # the copy)
    if mat and B:
        flat = token_lists
        ptrs = np.arange(B, dtype=np.uint64) * np.uint64(4 * token_lists.shape[1]) + np.uint64(flat.ctypes.data)
    elif B:
        flat = np.concatenate(toks) if B > 1 else toks[0]
        offs = np.zeros(B, dtype=np.uint64)
        np.cumsum(lens[:-1], out=offs[1:])
        ptrs = offs * np.uint64(4) + np.uint64(flat.ctypes.data)
    else:
        ptrs = np.zeros(1, dtype=np.uint64)
    arr = ptrs.ctypes.data_as(ctypes.POINTER(_I32P))
    _ok(_lib().sgl_build_batch(tree, B, arr, lens.ctypes.data_as(_I64P), _ptr32(table), ld, _ptr32(seq),
                               _ptr32(pre), last.ctypes.data_as(_I64P), groups), "sgl_build_batch")
    return {"req_to_token": table, "seq_lens": seq, "prefix_lens": pre, "last_nodes": last}


def sgl_batch_append(tree, req_to_token, seq_lens, groups=None):
    """One decode step of a running batch, in place: row r of `req_to_token`
    ([B, ld] int32, C-contiguous, writeable) gets a slot at position
    seq_lens[r] and `seq_lens` ([B] int32) grows by one; `groups` (the
    batch's prefix groups, or None) is updated to match."""
    B = seq_lens.shape[0] if isinstance(seq_lens, np.ndarray) else -1
    table = _out_i32(req_to_token, (B, req_to_token.shape[-1]), "req_to_token")
    seq = _out_i32(seq_lens, (B,), "seq_lens")
    _ok(_lib().sgl_batch_append(tree, B, _ptr32(table), table.shape[1], _ptr32(seq), groups), "sgl_batch_append")


def sgl_tree_cache_finished(tree, last, tokens, row, length):
    """Cache a finished request's sequence and release it; returns the
    duplicate tokens freed."""
    t, r = _i32(tokens), _i32(row)
    if t.shape[0] < length or r.shape[0] < length:
        raise ValueError("tokens and row must hold `length` entries")
    dup = ctypes.c_int64(0)
    _ok(_lib().sgl_tree_cache_finished(tree, int(last), _ptr32(t), _ptr32(r), int(length), ctypes.byref(dup)),
        "sgl_tree_cache_finished")
    return dup.value


def sgl_tree_cache_finished_batch(tree, tokens, out):
    """sgl_tree_cache_finished for every request of a batch: `tokens` is a
    [B, cap] int32 token matrix (row r holds at least out["seq_lens"][r]
    tokens) or a list of B token arrays; `out` a sgl_build_batch result
    (its dict), possibly advanced by sgl_batch_append."""
    last = np.ascontiguousarray(out["last_nodes"], dtype=np.int64)
    table = np.ascontiguousarray(out["req_to_token"], dtype=np.int32)
    seq = _i32(out["seq_lens"])
    B = len(seq)
    if isinstance(tokens, np.ndarray) and tokens.ndim == 2:
        if tokens.dtype != np.int32 or not tokens.flags.c_contiguous or tokens.shape[0] != B:
            raise ValueError("a token matrix must be C-contiguous int32 with B rows")
        if B and int(seq.max()) > tokens.shape[1]:
            raise ValueError("a row of the token matrix is shorter than its length")
        keep = tokens
        ptrs = np.arange(B, dtype=np.uint64) * np.uint64(4 * tokens.shape[1]) + np.uint64(tokens.ctypes.data)
    else:
        keep = [_i32(x) for x in tokens]
        if len(keep) != B or any(k.shape[0] < n for k, n in zip(keep, seq)):
            raise ValueError("one token array of at least seq_lens[r] tokens per request")
        ptrs = np.array([k.ctypes.data for k in keep] or [0], dtype=np.uint64)
    arr = ptrs.ctypes.data_as(ctypes.POINTER(_I32P))
    _ok(_lib().sgl_tree_cache_finished_batch(tree, B, arr, last.ctypes.data_as(_I64P), _ptr32(table), table.shape[1],
                                             _ptr32(seq)), "sgl_tree_cache_finished_batch")
    del keep


def sgl_tree_finish(tree, last, row, length):
    r = _i32(row)
    _ok(_lib().sgl_tree_finish(tree, int(last), _ptr32(r), int(length)), "sgl_tree_finish")


def sgl_tree_finish_batch(tree, out):
    """Finish every request of a sgl_build_batch result (its dict)."""
    last = np.ascontiguousarray(out["last_nodes"], dtype=np.int64)
    table = np.ascontiguousarray(out["req_to_token"], dtype=np.int32)
    seq = _i32(out["seq_lens"])
    _ok(_lib().sgl_tree_finish_batch(tree, len(seq), last.ctypes.data_as(_I64P), _ptr32(table), table.shape[1],
                                     _ptr32(seq)), "sgl_tree_finish_batch")


def sgl_groups_create():
    h = _P()
    _ok(_lib().sgl_groups_create(ctypes.byref(h)), "sgl_groups_create")
    return h


def sgl_groups_destroy(groups):
    _lib().sgl_groups_destroy(groups)


def sgl_groups_view(groups):
    """The groups as a ctypes view (valid while `groups` is unchanged)."""
    v = SglPrefixGroups()
    _ok(_lib().sgl_groups_view(groups, ctypes.byref(v)), "sgl_groups_view")
    return v


def groups_as_numpy(view):
    n, m = view.num_segments, view.num_members

    def arr(p, k):
        return np.ctypeslib.as_array(p, shape=(k,)).copy() if k else np.zeros(0, dtype=np.int32)
    return {"seg_begin": arr(view.seg_begin, n), "seg_end": arr(view.seg_end, n), "seg_row": arr(view.seg_row, n),
            "seg_member_ptr": arr(view.seg_member_ptr, n + 1), "seg_members": arr(view.seg_members, m)}


def sgl_groups_from_table(req_to_token, seq_lens, groups):
    t, s = _i32(req_to_token), _i32(seq_lens)
    _ok(_lib().sgl_groups_from_table(_ptr32(t), t.shape[1], _ptr32(s), len(s), groups), "sgl_groups_from_table")


# ------------------------------------------------------------- attention
def make_params(dtype, batch, num_qo_heads, num_kv_heads, head_dim, num_slots, page_size=1, sm_scale=0.0,
                num_sms=0, host_prefix_lens=None, host_extend_lens=None, k_scale=1.0, v_scale=1.0):
    p = SglAttnParams()
    p.k_scale = k_scale
    p.v_scale = v_scale
    p.dtype = dtype
    p.batch = batch
    p.num_qo_heads = num_qo_heads
    p.num_kv_heads = num_kv_heads
    p.head_dim = head_dim
    p.page_size = page_size
    p.num_slots = num_slots
    p.sm_scale = sm_scale
    p.num_sms = num_sms
    p._keep = []
    if host_prefix_lens is not None:
        a = _i32(host_prefix_lens)
        p._keep.append(a)
        p.host_prefix_lens = _ptr32(a)
    if host_extend_lens is not None:
        a = _i32(host_extend_lens)
        p._keep.append(a)
        p.host_extend_lens = _ptr32(a)
    return p


class Plan:
    """Owns an sgl_plan handle and its workspace size."""

    def __init__(self, handle, workspace_bytes):
        self.handle = handle
        self.workspace_bytes = workspace_bytes

    def __del__(self):
        if self.handle and _LIB is not None:
            _LIB.sgl_plan_destroy(self.handle)
            self.handle = None


def sgl_decode_plan(params, seq_lens, groups_view):
    s = _i32(seq_lens)
    h = _P()
    ws = ctypes.c_size_t()
    _ok(_lib().sgl_decode_plan(ctypes.byref(params), _ptr32(s), ctypes.byref(groups_view), ctypes.byref(h),
                               ctypes.byref(ws)), "sgl_decode_plan")
    return Plan(h, ws.value)


def sgl_plan_info(plan):
    i = SglPlanInfo()
    _ok(_lib().sgl_plan_info(plan.handle, ctypes.byref(i)), "sgl_plan_info")
    return {k: getattr(i, k) for k, _ in SglPlanInfo._fields_}


def sgl_plan_upload(plan, workspace, stream=None):
    _ok(_lib().sgl_plan_upload(plan.handle, _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
                               _stream(stream)), "sgl_plan_upload")


def sgl_decode_attn(q, k_pool, v_pool, req_to_token, seq_lens, plan, o, lse, workspace, stream=None):
    _ok(_lib().sgl_decode_attn(_dev(q, "q"), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"),
                               _dev(req_to_token, "req_to_token"), req_to_token.shape[1], _dev(seq_lens, "seq_lens"),
                               plan.handle, _dev(o, "o"), _dev(lse, "lse"), _dev(workspace, "workspace"),
                               workspace.numel() * workspace.element_size(), _stream(stream)), "sgl_decode_attn")


def _host(t, what):
    import torch
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError("%s must be a host tensor" % what)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % what)
    return ctypes.c_void_p(t.data_ptr())


def _in_region(t, region, what):
    """A CUDA tensor that lies inside the device tensor `region`."""
    p = _dev(t, what)
    lo, n = region.data_ptr(), region.numel() * region.element_size()
    if not (lo <= t.data_ptr() and t.data_ptr() + t.numel() * t.element_size() <= lo + n):
        raise ValueError("%s must lie inside its staging tensor" % what)
    return p


def sgl_decode_step(in_host, in_dev, q, k_pool, v_pool, req_to_token, seq_lens, plan, o, lse, out_dev, out_host,
                    workspace, stream=None):
    """One decode step from host memory: in_host -> in_dev (which holds q,
    req_to_token and seq_lens), the decode, out_dev (holding o and lse) ->
    out_host, queued on the stream by one library call."""
    nin = in_host.numel() * in_host.element_size()
    nout = out_host.numel() * out_host.element_size()
    if in_dev.numel() * in_dev.element_size() != nin or out_dev.numel() * out_dev.element_size() != nout:
        raise ValueError("staging tensors differ in size from their host buffers")
    _ok(_lib().sgl_decode_step(_host(in_host, "in_host"), _dev(in_dev, "in_dev"), nin,
                               _in_region(q, in_dev, "q"), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"),
                               _in_region(req_to_token, in_dev, "req_to_token"), req_to_token.shape[1],
                               _in_region(seq_lens, in_dev, "seq_lens"), plan.handle,
                               _in_region(o, out_dev, "o"), _in_region(lse, out_dev, "lse"), _dev(out_dev, "out_dev"),
                               _host(out_host, "out_host"), nout, _dev(workspace, "workspace"),
                               workspace.numel() * workspace.element_size(), _stream(stream)), "sgl_decode_step")


def make_mla_params(batch, num_qo_heads, num_slots, latent_dim=512, rope_dim=64, page_size=1, sm_scale=0.0,
                    num_sms=0):
    p = SglMlaParams()
    p.batch = batch
    p.num_qo_heads = num_qo_heads
    p.latent_dim = latent_dim
    p.rope_dim = rope_dim
    p.num_slots = num_slots
    p.page_size = page_size
    p.sm_scale = sm_scale
    p.num_sms = num_sms
    return p


def sgl_mla_decode_plan(params, seq_lens, groups_view):
    s = _i32(seq_lens)
    h = _P()
    ws = ctypes.c_size_t()
    _ok(_lib().sgl_mla_decode_plan(ctypes.byref(params), _ptr32(s), ctypes.byref(groups_view), ctypes.byref(h),
                                   ctypes.byref(ws)), "sgl_mla_decode_plan")
    return Plan(h, ws.value)


def sgl_mla_decode_attn(q, kv_pool, req_to_token, seq_lens, plan, o, lse, workspace, stream=None):
    _ok(_lib().sgl_mla_decode_attn(_dev(q, "q"), _dev(kv_pool, "kv_pool"), _dev(req_to_token, "req_to_token"),
                                   req_to_token.shape[1], _dev(seq_lens, "seq_lens"), plan.handle, _dev(o, "o"),
                                   _dev(lse, "lse"), _dev(workspace, "workspace"),
                                   workspace.numel() * workspace.element_size(), _stream(stream)),
        "sgl_mla_decode_attn")


def sgl_extend_workspace_bytes(params):
    b = ctypes.c_size_t()
    _ok(_lib().sgl_extend_workspace_bytes(ctypes.byref(params), ctypes.byref(b)), "sgl_extend_workspace_bytes")
    return b.value


def sgl_extend_attn(q_new, k_pool, v_pool, req_to_token, prefix_lens, extend_lens, params, o, lse, workspace,
                    stream=None):
    _ok(_lib().sgl_extend_attn(_dev(q_new, "q_new"), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"),
                               _dev(req_to_token, "req_to_token"), req_to_token.shape[1],
                               _dev(prefix_lens, "prefix_lens"), _dev(extend_lens, "extend_lens"),
                               ctypes.byref(params), _dev(o, "o"), _dev(lse, "lse"), _dev(workspace, "workspace"),
                               workspace.numel() * workspace.element_size(), _stream(stream)), "sgl_extend_attn")


def sgl_extend_attn_kvwrite(q_new, k_new, v_new, k_pool, v_pool, req_to_token, prefix_lens, extend_lens, params, o,
                            lse, workspace, stream=None):
    _ok(_lib().sgl_extend_attn_kvwrite(_dev(q_new, "q_new"), _dev(k_new, "k_new"), _dev(v_new, "v_new"),
                                       _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"),
                                       _dev(req_to_token, "req_to_token"), req_to_token.shape[1],
                                       _dev(prefix_lens, "prefix_lens"), _dev(extend_lens, "extend_lens"),
                                       ctypes.byref(params), _dev(o, "o"), _dev(lse, "lse"),
                                       _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
                                       _stream(stream)), "sgl_extend_attn_kvwrite")


def sgl_check(workspace, stream=None):
    _ok(_lib().sgl_check(_dev(workspace, "workspace"), _stream(stream)), "sgl_check")


def sgl_decode_attn_noalloc(q, k_pool, v_pool, req_to_token, seq_lens, plan, o, lse, stream=None):
    """Decode with the library's fixed device scratch (for callers that cannot allocate)."""
    _ok(_lib().sgl_decode_attn_noalloc(_dev(q, "q"), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"),
                                       _dev(req_to_token, "req_to_token"), req_to_token.shape[1],
                                       _dev(seq_lens, "seq_lens"), plan.handle, _dev(o, "o"), _dev(lse, "lse"),
                                       _stream(stream)), "sgl_decode_attn_noalloc")
