"""MLA decode planner on the host (no GPU): work-item and merge-list
invariants, rejected shapes and plan kinds."""

import ctypes

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
    assert info["num_wide_items"] == 0 and info["chunk_tokens"] % 32 == 0


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
