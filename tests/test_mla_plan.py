"""MLA decode planner on the host (no GPU): work-item and merge-list
invariants, rejected shapes and plan kinds."""

import ctypes
import time

import numpy as np
import pytest

import radixattention_prefix_shared_radix_gb300 as sgl
import workloads as W
from tests._harness import Case


@pytest.fixture(scope="module", params=["mla_decode_small", "mla_decode_h128_small"])
def case(request):
    w = W.get(request.param)
    c = Case(request.param, pool=W.make_mla_pool(w) + (None,))
    yield c
    c.close()


def _plan(case, **kw):
    w = case.w
    p = sgl.make_mla_params(case.B, w.Hq, case.S, page_size=w.page_size, num_sms=kw.pop("num_sms", 152), **kw)
    return sgl.sgl_mla_decode_plan(p, case.out["seq_lens"], sgl.sgl_groups_view(case.groups))


@pytest.mark.parametrize("num_sms", [1, 3, 152])
def test_every_partial_row_group_is_merged_once(case, num_sms):
    w = case.w
    Gp = min(w.Hq, 64)
    info = sgl.sgl_plan_info(_plan(case, num_sms=num_sms))
    assert info["num_partial_rows"] == info["num_merge_entries"] * Gp
    # tile pieces are two units each (two CTAs, one per output half)
    assert info["num_wide_items"] % 2 == 0 and info["num_wide_items"] <= info["num_items"]
    assert info["chunk_tokens"] % 32 == 0


def test_segments_with_two_full_units_become_tiles(case):
    # a segment that holds two full 64-row units (members x heads of a head
    # group) is read by a tcgen05 tile pair; these workloads have such
    # segments (a shared prefix; or one request's two head groups at Hq 128)
    info = sgl.sgl_plan_info(_plan(case))
    assert info["num_wide_items"] > 0


def test_items_cover_every_member_once_per_position(case):
    # rows x positions summed over items = sum over requests of
    # seq_len x query heads (each member block covers its members' heads)
    info = sgl.sgl_plan_info(_plan(case))
    g = sgl.groups_as_numpy(sgl.sgl_groups_view(case.groups))
    entries = sum(int(m1 - m0) for m0, m1 in zip(g["seg_member_ptr"][:-1], g["seg_member_ptr"][1:]))
    Hg = max(1, case.w.Hq // 64)
    assert info["num_merge_entries"] >= entries * Hg


@pytest.mark.parametrize("field,value", [("latent_dim", 256), ("rope_dim", 32), ("num_qo_heads", 8),
                                         ("num_qo_heads", 48)])
def test_unsupported_shapes(case, field, value):
    w = case.w
    p = sgl.make_mla_params(case.B, w.Hq, case.S, num_sms=152)
    setattr(p, field, value)
    with pytest.raises(sgl.SglError) as e:
        sgl.sgl_mla_decode_plan(p, case.out["seq_lens"], sgl.sgl_groups_view(case.groups))
    assert e.value.status == -3


def test_plan_kinds_are_not_interchangeable(case):
    lib = sgl._lib()
    mla = _plan(case)
    # an MLA plan into the GQA decode, and a GQA plan into the MLA decode:
    # both rejected before any device access
    st = lib.sgl_decode_attn(None, None, None, None, 0, None, mla.handle, None, None, None, 0, None)
    assert st == -1
    gqa_case = Case("llama3_8b_decode_small")
    try:
        w = gqa_case.w
        p = sgl.make_params(sgl.SGL_DTYPE_BF16, gqa_case.B, w.Hq, w.Hkv, w.d, gqa_case.S, w.page_size, num_sms=152)
        gqa = sgl.sgl_decode_plan(p, gqa_case.out["seq_lens"], sgl.sgl_groups_view(gqa_case.groups))
        st = lib.sgl_mla_decode_attn(None, None, None, 0, None, gqa.handle, None, None, None, 0, None)
        assert st == -1
    finally:
        gqa_case.close()


def test_cost_model_plan_is_deterministic_and_bounded():
    """The piece length is chosen by simulating the schedule: the same
    inputs give the same plan, the item count stays within a few waves
    (partial rows cost merge traffic), and the longest piece is whole
    32-position blocks."""
    w = W.get("mla_decode")
    b = W.make_batch(w, 0)
    seqs = b.all_tokens()
    S = 1 << 20
    tree = sgl.sgl_tree_create(S, w.page_size, np.arange(S, dtype=np.int32))
    groups = sgl.sgl_groups_create()
    try:
        out = sgl.sgl_build_batch(tree, seqs, groups=groups)
        infos = []
        for sms in (152, 152, 132, 16):
            p = sgl.make_mla_params(len(seqs), w.Hq, S, num_sms=sms)
            infos.append((sms, sgl.sgl_plan_info(sgl.sgl_mla_decode_plan(p, out["seq_lens"],
                                                                          sgl.sgl_groups_view(groups)))))
        assert infos[0][1] == infos[1][1]
        for sms, info in infos:
            assert info["chunk_tokens"] % 32 == 0 and info["chunk_tokens"] >= 64
            assert sms // 2 <= info["num_items"] <= 3 * sms + 80, (sms, info)
    finally:
        sgl.sgl_groups_destroy(groups)
        sgl.sgl_tree_destroy(tree)


def test_huge_sm_count_and_one_token_segments(case):
    w = case.w
    t0 = time.perf_counter()
    info = sgl.sgl_plan_info(_plan(case, num_sms=1 << 20))
    assert time.perf_counter() - t0 < 5.0
    assert info["num_items"] > 0
    # every request one token long, no sharing: one item per (member block, head group)
    seqs = [[int(t)] for t in range(7)]
    S = 1 << 12
    tree = sgl.sgl_tree_create(S, 1, np.arange(S, dtype=np.int32))
    groups = sgl.sgl_groups_create()
    try:
        out = sgl.sgl_build_batch(tree, seqs, groups=groups)
        p = sgl.make_mla_params(len(seqs), w.Hq, S, num_sms=152)
        info = sgl.sgl_plan_info(sgl.sgl_mla_decode_plan(p, out["seq_lens"], sgl.sgl_groups_view(groups)))
        Hg = max(1, w.Hq // 64)
        assert info["num_items"] == len(seqs) * Hg
        assert info["num_merge_entries"] == len(seqs) * Hg
    finally:
        sgl.sgl_groups_destroy(groups)
        sgl.sgl_tree_destroy(tree)
