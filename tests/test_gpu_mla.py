"""MLA grouped decode on the GPU vs the float64 MLA oracle (through the C ABI).

Element by element on the small MLA workloads (16 and 128 query heads,
several SM counts so that segments are cut into different chunks), with a
model scale other than the default, an empty request, and at the full
workload size on every request.  The oracle reads every request's context
with no sharing.  Tolerances: bf16 O max-abs 2e-2, LSE 1e-3.
"""

import math

import numpy as np
import pytest
import torch

import radixattention_prefix_shared_radix_gb300 as sgl
import workloads as W
from oracle.mla import mla_decode_attention
from tests._harness import BF16_LSE_TOL, BF16_O_TOL, Case, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from radixattention_prefix_shared_radix_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _mla_case(name, seqs=None):
    w = W.get(name)
    return Case(name, pool=W.make_mla_pool(w) + (None,), seqs=seqs)


def _run(case, num_sms=0, sm_scale=0.0, kv=None):
    w = case.w
    p = sgl.make_mla_params(case.B, w.Hq, case.S, page_size=w.page_size, sm_scale=sm_scale, num_sms=num_sms)
    plan = sgl.sgl_mla_decode_plan(p, case.out["seq_lens"], sgl.sgl_groups_view(case.groups))
    ws = torch.zeros(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    sgl.sgl_plan_upload(plan, ws)
    qd = case.q_host().cuda()
    kvd = case.K.cuda() if kv is None else kv
    table = torch.from_numpy(case.out["req_to_token"]).cuda()
    seq = torch.from_numpy(case.out["seq_lens"]).cuda()
    o = torch.empty(case.B, w.Hq, w.dv, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(case.B, w.Hq, dtype=torch.float32, device="cuda")
    sgl.sgl_mla_decode_attn(qd, kvd, table, seq, plan, o, lse, ws)
    sgl.sgl_check(ws)
    info = sgl.sgl_plan_info(plan)
    del plan
    return o.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64), info


def _oracle(case, sm_scale=None, requests=None):
    return mla_decode_attention(case.oracle_q(), W.RowView(case.K), case.oracle_table, case.out["seq_lens"],
                                case.w.dv, sm_scale=sm_scale, requests=requests)


@pytest.mark.parametrize("name", ["mla_decode_small", "mla_decode_h128_small"])
@pytest.mark.parametrize("num_sms", [0, 1, 5])
def test_mla_small_elementwise(name, num_sms):
    case = _mla_case(name)
    try:
        O, L, info = _run(case, num_sms=num_sms)
        Oref, Lref = _oracle(case)
        assert_close(O, L, Oref, Lref, BF16_O_TOL, BF16_LSE_TOL)
        assert info["num_items"] > 0
    finally:
        case.close()


def test_mla_model_scale():
    case = _mla_case("mla_decode_small")
    try:
        sc = 1.0 / math.sqrt(192.0)
        O, L, _ = _run(case, sm_scale=sc)
        Oref, Lref = _oracle(case, sm_scale=sc)
        assert_close(O, L, Oref, Lref, BF16_O_TOL, BF16_LSE_TOL)
    finally:
        case.close()


def test_mla_edge_batch():
    """Empty context, one-token contexts, a request that is a prefix of
    another, identical requests (shared prefixes of 2..4 members)."""
    w = W.get("mla_decode_small")
    rng = np.random.default_rng(78)
    base = list(rng.integers(0, 32000, size=250))
    seqs = [base, [], base[:1], base[:100], list(base), base[:100] + [5, 6, 7], [9] * 40, [9]]
    q = rng.standard_normal((len(seqs), w.Hq, w.d), dtype=np.float32)
    case = Case(None, workload=w, seqs=seqs, q=q, pool=W.make_mla_pool(w) + (None,))
    try:
        O, L, _ = _run(case)
        assert np.all(O[1] == 0) and np.all(np.isneginf(L[1]))
        Oref, Lref = _oracle(case)
        assert_close(O, L, Oref, Lref, BF16_O_TOL, BF16_LSE_TOL)
    finally:
        case.close()


def test_mla_full_size():
    case = _mla_case("mla_decode")
    try:
        O, L, info = _run(case)
        Oref, Lref = _oracle(case)
        do, dl = assert_close(O, L, Oref, Lref, BF16_O_TOL, BF16_LSE_TOL)
        print("mla_decode: O max-abs %.3g, LSE max-abs %.3g, items %d" % (do, dl, info["num_items"]))
    finally:
        case.close()


def test_mla_out_of_pool_slot_is_reported_not_read():
    case = _mla_case("mla_decode_small")
    try:
        w = case.w
        p = sgl.make_mla_params(case.B, w.Hq, case.S)
        plan = sgl.sgl_mla_decode_plan(p, case.out["seq_lens"], sgl.sgl_groups_view(case.groups))
        ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
        sgl.sgl_plan_upload(plan, ws)
        table = torch.from_numpy(case.out["req_to_token"]).cuda()
        # a position of request 3's own suffix (shared positions are read
        # from the segment's representative row)
        table[3, int(case.out["seq_lens"][3]) - 1] = case.S + 11
        qd = case.q_host().cuda()
        kvd = case.K.cuda()
        o = torch.empty(case.B, w.Hq, w.dv, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(case.B, w.Hq, dtype=torch.float32, device="cuda")
        seq = torch.from_numpy(case.out["seq_lens"]).cuda()
        sgl.sgl_mla_decode_attn(qd, kvd, table, seq, plan, o, lse, ws)
        with pytest.raises(sgl.SglError) as e:
            sgl.sgl_check(ws)
        assert e.value.status == -5
        sgl.sgl_check(ws)          # the word was cleared
        # a plan that disagrees with the device seq_lens is reported too
        seq[0] = 1
        sgl.sgl_mla_decode_attn(qd, kvd, torch.from_numpy(case.out["req_to_token"]).cuda(), seq, plan, o, lse, ws)
        with pytest.raises(sgl.SglError):
            sgl.sgl_check(ws)
        del plan
    finally:
        case.close()
