"""Shared set-up for the GPU parity tests: seeded inputs -> native tables ->
CUDA kernels, and the oracle on its own tables from the same inputs."""

import numpy as np
import torch

import radixattention_prefix_shared_radix_gb300 as sgl
import workloads as W
from oracle.tree import RadixTrie, build_batch

BF16_O_TOL, BF16_LSE_TOL = 2e-2, 1e-3
F32_O_TOL, F32_LSE_TOL = 1e-4, 1e-4


def tolerances(w):
    return (F32_O_TOL, F32_LSE_TOL) if w.dtype == "f32" else (BF16_O_TOL, BF16_LSE_TOL)


class Case:
    """One workload instance with native and oracle tables built side by side."""

    def __init__(self, name, instance=0, pool=None, seqs=None, workload=None, q=None):
        self.w = workload or W.get(name)
        w = self.w
        self.b = W.make_batch(w, instance)
        if q is not None:
            self.b.q = q
        if pool is None:
            pool = W.make_pool(w)
        self.order, self.K, self.V = pool
        self.S = self.K.shape[0]
        self.tree = sgl.sgl_tree_create(self.S, w.page_size, self.order)
        self.trie = RadixTrie(self.S, w.page_size, self.order)
        self.groups = sgl.sgl_groups_create()
        if w.kind == "extend":
            warm = [self.b.cached_tokens(r) for r in range(len(self.b.req_chain))]
            out = sgl.sgl_build_batch(self.tree, warm)
            for r in range(len(warm)):
                sgl.sgl_tree_finish(self.tree, int(out["last_nodes"][r]), out["req_to_token"][r], len(warm[r]))
            _, lasts, _ = build_batch(self.trie, warm)
            for n in lasts:
                self.trie.unlock(n)
        self.seqs = seqs if seqs is not None else self.b.all_tokens()
        self.out = sgl.sgl_build_batch(self.tree, self.seqs, groups=self.groups)
        rows, _, _ = build_batch(self.trie, self.seqs)
        ld = self.out["req_to_token"].shape[1]
        self.oracle_table = np.full((len(rows), ld), -1, dtype=np.int64)
        for r, row in enumerate(rows):
            self.oracle_table[r, :len(row)] = row
        self.B = len(self.seqs)

    def close(self):
        sgl.sgl_groups_destroy(self.groups)
        sgl.sgl_tree_destroy(self.tree)

    # device copies ------------------------------------------------------
    def device_pool(self):
        return self.K.cuda(), self.V.cuda()

    def q_host(self):
        return W.to_dtype(self.w, self.b.q)

    def params(self, **kw):
        w = self.w
        dt = sgl.SGL_DTYPE_F32 if w.dtype == "f32" else sgl.SGL_DTYPE_BF16
        return sgl.make_params(dt, self.B, w.Hq, w.Hkv, w.d, self.S, w.page_size, **kw)

    def oracle_q(self):
        return self.q_host().double().numpy()


def run_decode(case, kpool, vpool, num_sms=0, q=None):
    """GPU decode through the C ABI; returns (O float64 numpy, LSE numpy)."""
    p = case.params(num_sms=num_sms)
    plan = sgl.sgl_decode_plan(p, case.out["seq_lens"], sgl.sgl_groups_view(case.groups))
    ws = torch.zeros(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    sgl.sgl_plan_upload(plan, ws)
    qd = (q if q is not None else case.q_host()).cuda()
    table = torch.from_numpy(case.out["req_to_token"]).cuda()
    seq = torch.from_numpy(case.out["seq_lens"]).cuda()
    o = torch.empty_like(qd)
    lse = torch.empty(case.B, case.w.Hq, dtype=torch.float32, device="cuda")
    sgl.sgl_decode_attn(qd, kpool, vpool, table, seq, plan, o, lse, ws)
    sgl.sgl_check(ws)
    return o.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64)


def run_extend(case, kpool, vpool):
    pre = case.out["prefix_lens"]
    ext = case.out["seq_lens"] - pre
    p = case.params(host_prefix_lens=pre, host_extend_lens=ext)
    ws = torch.zeros(sgl.sgl_extend_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    qd = case.q_host().cuda()
    table = torch.from_numpy(case.out["req_to_token"]).cuda()
    o = torch.empty_like(qd)
    lse = torch.empty(qd.shape[0], case.w.Hq, dtype=torch.float32, device="cuda")
    sgl.sgl_extend_attn(qd, kpool, vpool, table, torch.from_numpy(pre).cuda(), torch.from_numpy(ext).cuda(), p, o,
                        lse, ws)
    sgl.sgl_check(ws)
    return o.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64), pre, ext


def assert_close(O, L, Oref, Lref, otol, ltol, rows=None):
    if rows is not None:
        O, L, Oref, Lref = O[rows], L[rows], Oref[rows], Lref[rows]
    finite = np.isfinite(Lref)
    assert np.array_equal(np.isfinite(L), finite), "LSE -inf pattern differs"
    do = np.abs(O - Oref).max() if O.size else 0.0
    dl = np.abs(L[finite] - Lref[finite]).max() if finite.any() else 0.0
    assert do <= otol, "O max-abs error %.3g > %.3g" % (do, otol)
    assert dl <= ltol, "LSE max-abs error %.3g > %.3g" % (dl, ltol)
    return do, dl


def full_and_sampled_rows(ext, full, seed, picks):
    """Every new-token row of the requests in ``full`` (all query heads: every
    tile position, causal edge and K/V block of those requests), plus, for the
    other requests, the first and last rows, the rows at ``picks`` and four
    random ones."""
    starts = np.concatenate([[0], np.cumsum(ext)[:-1]])
    rng = np.random.default_rng(seed)
    rows = []
    for r, (s, e) in enumerate(zip(starts, ext)):
        if r in full:
            rows += list(range(int(s), int(s + e)))
        else:
            rows += [int(s), int(s + e - 1)] + [int(s + p) for p in picks if p < e]
            rows += [int(s + x) for x in rng.integers(0, e, 4)]
    return sorted(set(rows))
