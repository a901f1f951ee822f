"""Decode through the no-allocation entry point (GPU).

Some callers cannot allocate device memory (a serving loop whose memory
another allocator owns under a fixed budget, a path that must not risk
cudaMalloc synchronizing the device).  For them the library offers
sgl_decode_attn_noalloc, which uses a fixed scratch array in its own device
image instead of a caller workspace.  This test calls it through the C ABI
twice in a row and checks both results against sgl_decode_attn with a
caller workspace, that the calls leave the torch allocator's device memory
unchanged, and that a plan too large for the scratch, or another argument
error, is refused.
"""

import numpy as np
import pytest
import torch

import radixattention_prefix_shared_radix_gb300 as sgl
import workloads as W
from tests._harness import Case, tolerances

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from radixattention_prefix_shared_radix_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def test_noalloc_matches_workspace_decode_twice():
    case = Case("llama3_8b_decode_small")
    try:
        kd, vd = case.device_pool()
        p = case.params()
        plan = sgl.sgl_decode_plan(p, case.out["seq_lens"], sgl.sgl_groups_view(case.groups))
        q = case.q_host().cuda()
        table = torch.from_numpy(case.out["req_to_token"]).cuda()
        seq = torch.from_numpy(case.out["seq_lens"]).cuda()
        ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
        sgl.sgl_plan_upload(plan, ws)
        o_ref = torch.empty_like(q)
        lse_ref = torch.empty(case.B, case.w.Hq, dtype=torch.float32, device="cuda")
        sgl.sgl_decode_attn(q, kd, vd, table, seq, plan, o_ref, lse_ref, ws)
        sgl.sgl_check(ws)
        otol, ltol = tolerances(case.w)
        outs = [(torch.full_like(q, float("nan")),
                 torch.full((case.B, case.w.Hq), float("nan"), dtype=torch.float32, device="cuda")) for _ in range(2)]
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
        for o, lse in outs:
            sgl.sgl_decode_attn_noalloc(q, kd, vd, table, seq, plan, o, lse)
            torch.cuda.synchronize()
            assert (torch.cuda.memory_allocated(), torch.cuda.memory_reserved()) == before
            assert torch.isfinite(lse).all()
            assert (o.float() - o_ref.float()).abs().max().item() <= otol
            assert (lse - lse_ref).abs().max().item() <= ltol
    finally:
        case.close()


def test_noalloc_rejects_plan_beyond_scratch():
    # many small chunks: a plan whose partial buffers exceed the 64 MiB scratch
    B, L = 256, 4096
    seqs = [list(np.random.default_rng(r).integers(0, 32000, size=L)) for r in range(B)]
    tree = sgl.sgl_tree_create(1 << 21, 1)
    g = sgl.sgl_groups_create()
    try:
        out = sgl.sgl_build_batch(tree, seqs, groups=g)
        p = sgl.make_params(sgl.SGL_DTYPE_BF16, B, 32, 8, 128, 1 << 21, 1, num_sms=100000)
        plan = sgl.sgl_decode_plan(p, out["seq_lens"], sgl.sgl_groups_view(g))
        assert plan.workspace_bytes > 64 << 20
        dummy = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
        table = torch.zeros(1, dtype=torch.int32, device="cuda")
        with pytest.raises(sgl.SglError) as e:
            sgl.sgl_decode_attn_noalloc(dummy, dummy, dummy, table.view(1, 1), table, plan, dummy, dummy.float())
        assert e.value.status == -7
    finally:
        sgl.sgl_groups_destroy(g)
        sgl.sgl_tree_destroy(tree)


def test_noalloc_refuses_a_bad_call_before_gpu_work():
    """An MLA plan, or a slot table narrower than the plan's positions, is
    refused with SGL_ERR_INVALID_ARG by the argument checks."""
    case = Case("llama3_8b_decode_small")
    try:
        kd, vd = case.device_pool()
        plan = sgl.sgl_decode_plan(case.params(), case.out["seq_lens"], sgl.sgl_groups_view(case.groups))
        q = case.q_host().cuda()
        seq = torch.from_numpy(case.out["seq_lens"]).cuda()
        o = torch.empty_like(q)
        lse = torch.empty(case.B, case.w.Hq, dtype=torch.float32, device="cuda")
        narrow = torch.from_numpy(np.ascontiguousarray(case.out["req_to_token"][:, :1])).cuda()
        with pytest.raises(sgl.SglError) as e:
            sgl.sgl_decode_attn_noalloc(q, kd, vd, narrow, seq, plan, o, lse)
        assert e.value.status == -1
    finally:
        case.close()
