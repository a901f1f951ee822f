"""Decode planner invariants on the host (no GPU): the plan is host code, so
its counts can be checked here against the batch's prefix groups."""

import pytest

import radixattention_prefix_shared_radix_gb300 as sgl
from tests._harness import Case


@pytest.fixture(scope="module")
def case():
    c = Case("llama3_8b_decode_small")
    yield c
    c.close()


def _plan(case, dtype, **kw):
    w = case.w
    p = sgl.make_params(dtype, case.B, w.Hq, w.Hkv, w.d, case.S, w.page_size, num_sms=152, **kw)
    plan = sgl.sgl_decode_plan(p, case.out["seq_lens"], sgl.sgl_groups_view(case.groups))
    return sgl.sgl_plan_info(plan)


def test_every_partial_row_group_is_merged_once(case):
    G = case.w.Hq // case.w.Hkv
    for dt, kw in ((sgl.SGL_DTYPE_BF16, {}), (sgl.SGL_DTYPE_BF16_FP8KV, dict(k_scale=0.5, v_scale=0.25))):
        info = _plan(case, dt, **kw)
        assert info["num_partial_rows"] == info["num_merge_entries"] * G


def test_fp8_pool_plans_like_bf16(case):
    # the batch shares a long prefix among more members than a streaming
    # warp's 8 query rows: tensor-core tiles for it, with either pool type
    # (the plan depends on the batch, not on the pool's element type)
    b = _plan(case, sgl.SGL_DTYPE_BF16)
    f = _plan(case, sgl.SGL_DTYPE_BF16_FP8KV, k_scale=0.5, v_scale=0.25)
    assert b["num_wide_items"] > 0
    for k in ("num_items", "num_wide_items", "num_partial_rows", "num_merge_entries", "chunk_tokens"):
        assert b[k] == f[k], k


@pytest.mark.parametrize("ks,vs", [(0.0, 1.0), (1.0, -1.0)])
def test_fp8_scales_must_be_positive(case, ks, vs):
    with pytest.raises(sgl.SglError):
        _plan(case, sgl.SGL_DTYPE_BF16_FP8KV, k_scale=ks, v_scale=vs)


def test_a_piece_takes_at_most_eight_member_requests():
    """G = 1 and 2: a segment of 9..16 members has at most 16 query rows per
    KV head but more members than a streaming piece carries, so it is
    planned on tiles."""
    import workloads as W
    for Hq, Hkv, n, wide in ((8, 8, 12, True), (8, 8, 8, False), (16, 8, 12, True), (16, 8, 8, False)):
        w = W.Workload("members", 2, "decode", "bf16", Hq, Hkv, 128, 1,
                       ("star", dict(n=n, prefix=150, suffix=(1, 90))), num_slots=4096)
        c = Case(None, workload=w)
        try:
            info = _plan(c, sgl.SGL_DTYPE_BF16)
            assert (info["num_wide_items"] > 0) == wide, (Hq, Hkv, n, info)
        finally:
            c.close()
