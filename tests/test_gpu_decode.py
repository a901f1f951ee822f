"""Decode attention on the GPU vs the float64 oracle (through the C ABI).

Element by element on scaled-down shapes of every decode workload and on
edge cases; at the full workload sizes on every request.  The oracle runs
on its own trie's tables (bit-identical to the native ones, checked on CPU)
with no sharing, so agreement also shows that reading each shared segment
once gives the unshared result.  Tolerances: bf16 O max-abs 2e-2, LSE 1e-3;
fp32 O and LSE 1e-4.
"""

import numpy as np
import pytest
import torch

import radixattention_prefix_shared_radix_gb300 as sgl
import workloads as W
from oracle.attention import decode_attention
from tests._harness import Case, assert_close, full_and_sampled_rows, run_decode, tolerances

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from radixattention_prefix_shared_radix_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _check(case, num_sms=0, requests=None):
    kd, vd = case.device_pool()
    O, L = run_decode(case, kd, vd, num_sms=num_sms)
    Oref, Lref = decode_attention(case.oracle_q(), W.RowView(case.K), W.RowView(case.V), case.oracle_table,
                                  case.out["seq_lens"], requests=requests)
    return assert_close(O, L, Oref, Lref, *tolerances(case.w), rows=requests)


@pytest.mark.parametrize("name", ["tiny_fp32", "llama3_8b_decode_small", "fork_tree_small", "multiturn_small"])
def test_decode_small_workloads_elementwise(name):
    case = Case(name)
    try:
        _check(case)
    finally:
        case.close()


@pytest.mark.parametrize("num_sms", [1, 7, 152, 4000])
def test_decode_split_invariance(num_sms):
    """Different chunkings (from the planner's SM target) give the oracle's result."""
    case = Case("llama3_8b_decode_small")
    try:
        _check(case, num_sms=num_sms)
    finally:
        case.close()


SHAPES = [
    ("bf16", 8, 8, 64), ("bf16", 16, 8, 128), ("bf16", 64, 8, 128), ("bf16", 8, 4, 64),
    ("f32", 8, 1, 128), ("f32", 32, 8, 128), ("f32", 4, 2, 64),
]


@pytest.mark.parametrize("dtype,Hq,Hkv,d", SHAPES)
def test_decode_head_shapes(dtype, Hq, Hkv, d):
    w = W.Workload("shape", 2, "decode", dtype, Hq, Hkv, d, 1,
                   ("star", dict(n=6, prefix=77, suffix=(1, 150))), num_slots=2048)
    case = Case(None, workload=w)
    try:
        _check(case)
    finally:
        case.close()


@pytest.mark.parametrize("Hq,Hkv,d", [(8, 8, 128), (8, 8, 64), (16, 8, 128), (32, 8, 128)])
def test_decode_many_members_per_head(Hq, Hkv, d):
    """A prefix shared by 12 requests: 12 x G query rows per KV head (a
    streaming piece takes at most 8 member requests, so G = 1 and 2 put it
    on tiles, as G = 4 does)."""
    w = W.Workload("members", 2, "decode", "bf16", Hq, Hkv, d, 1,
                   ("star", dict(n=12, prefix=150, suffix=(1, 90))), num_slots=4096)
    case = Case(None, workload=w)
    try:
        _check(case)
    finally:
        case.close()


def test_decode_edge_batch():
    """Empty context, one-token contexts, a request that is a prefix of
    another, identical requests, a branch that starts at position 0."""
    w = W.get("llama3_8b_decode_small")
    rng = np.random.default_rng(77)
    base = list(rng.integers(0, 32000, size=300))
    seqs = [base, [], base[:1], base[:120], list(base), base[:120] + [5, 6, 7], [9] * 65, [9]]
    q = rng.standard_normal((len(seqs), w.Hq, w.d), dtype=np.float32)
    case = Case(None, workload=w, seqs=seqs, q=q)
    try:
        kd, vd = case.device_pool()
        O, L = run_decode(case, kd, vd)
        assert np.all(O[1] == 0) and np.all(np.isneginf(L[1]))
        Oref, Lref = decode_attention(case.oracle_q(), W.RowView(case.K), W.RowView(case.V), case.oracle_table,
                                      case.out["seq_lens"])
        assert_close(O, L, Oref, Lref, *tolerances(w))
    finally:
        case.close()


def test_decode_paged_edge():
    """page size 16 with contexts not a multiple of the page, shared and not."""
    w = W.get("multiturn_small")
    rng = np.random.default_rng(5)
    a = list(rng.integers(0, 32000, size=70))
    seqs = [a, a, a[:40] + [1, 2, 3], a[:16], a[:15], [7] * 33]
    q = rng.standard_normal((len(seqs), w.Hq, w.d), dtype=np.float32)
    case = Case(None, workload=w, seqs=seqs, q=q)
    try:
        kd, vd = case.device_pool()
        O, L = run_decode(case, kd, vd)
        Oref, Lref = decode_attention(case.oracle_q(), W.RowView(case.K), W.RowView(case.V), case.oracle_table,
                                      case.out["seq_lens"])
        assert_close(O, L, Oref, Lref, *tolerances(w))
    finally:
        case.close()


def test_decode_out_of_pool_slot_is_reported_not_read():
    case = Case("llama3_8b_decode_small")
    try:
        kd, vd = case.device_pool()
        p = case.params()
        plan = sgl.sgl_decode_plan(p, case.out["seq_lens"], sgl.sgl_groups_view(case.groups))
        ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
        sgl.sgl_plan_upload(plan, ws)
        table = torch.from_numpy(case.out["req_to_token"]).cuda()
        # a position of request 3's own suffix (shared prefix positions are
        # read from the segment's representative row, row 0)
        table[3, int(case.out["seq_lens"][3]) - 1] = case.S + 11
        qd = case.q_host().cuda()
        o = torch.empty_like(qd)
        lse = torch.empty(case.B, case.w.Hq, dtype=torch.float32, device="cuda")
        seq = torch.from_numpy(case.out["seq_lens"]).cuda()
        sgl.sgl_decode_attn(qd, kd, vd, table, seq, plan, o, lse, ws)
        with pytest.raises(sgl.SglError) as e:
            sgl.sgl_check(ws)
        assert e.value.status == -5
        sgl.sgl_check(ws)          # the word was cleared
        # a plan that disagrees with the device seq_lens is reported too
        seq[0] = 1
        sgl.sgl_decode_attn(qd, kd, vd, torch.from_numpy(case.out["req_to_token"]).cuda(), seq, plan, o, lse, ws)
        with pytest.raises(sgl.SglError):
            sgl.sgl_check(ws)
    finally:
        case.close()


def test_decode_rejects_malformed_groups():
    case = Case("llama3_8b_decode_small")
    try:
        view = sgl.sgl_groups_view(case.groups)
        p = case.params()
        seq = case.out["seq_lens"].copy()
        seq[2] += 1                          # request 2's segments no longer cover its context
        with pytest.raises(sgl.SglError) as e:
            sgl.sgl_decode_plan(p, seq, view)
        assert e.value.status == -1
    finally:
        case.close()


@pytest.mark.parametrize("name", ["llama3_8b_decode", "fork_tree", "multiturn", "multiturn_noshare"])
def test_decode_full_size(name):
    case = Case(name)
    try:
        do, dl = _check(case)
        print("%s: O max-abs %.3g, LSE max-abs %.3g" % (name, do, dl))
    finally:
        case.close()


def test_decode_rescale_path_with_growing_scores():
    """Large scores late in shared prefixes force the tensor-core tiles' running-max rescale."""
    w = W.get("llama3_8b_decode_small")
    order, K, V = W.make_pool(w)
    K = K.clone()
    K[::89] *= 30.0
    case = Case(None, workload=w, pool=(order, K, V))
    try:
        _check(case)
    finally:
        case.close()


@pytest.mark.parametrize("num_sms", [0, 3])
def test_decode_repeated_calls_share_one_upload(num_sms):
    """Calls after one plan upload give identical results: the kernel hands
    narrow pieces out from a run-time counter and restores it at the end of
    every call, so the tenth call without a new upload sees what the first
    saw.  Also captures three calls in a CUDA graph and replays it."""
    case = Case("fork_tree_small")
    try:
        kd, vd = case.device_pool()
        p = case.params(num_sms=num_sms)
        plan = sgl.sgl_decode_plan(p, case.out["seq_lens"], sgl.sgl_groups_view(case.groups))
        ws = torch.zeros(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
        sgl.sgl_plan_upload(plan, ws)
        qd = case.q_host().cuda()
        table = torch.from_numpy(case.out["req_to_token"]).cuda()
        seq = torch.from_numpy(case.out["seq_lens"]).cuda()
        o = torch.empty_like(qd)
        lse = torch.empty(case.B, case.w.Hq, dtype=torch.float32, device="cuda")
        sgl.sgl_decode_attn(qd, kd, vd, table, seq, plan, o, lse, ws)
        sgl.sgl_check(ws)
        o0, l0 = o.clone(), lse.clone()
        for _ in range(9):
            o.zero_()
            sgl.sgl_decode_attn(qd, kd, vd, table, seq, plan, o, lse, ws)
        sgl.sgl_check(ws)
        assert torch.equal(o, o0) and torch.equal(lse, l0)
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for _ in range(3):
                    sgl.sgl_decode_attn(qd, kd, vd, table, seq, plan, o, lse, ws)
        torch.cuda.current_stream().wait_stream(s)
        for _ in range(4):
            o.zero_()
            g.replay()
        torch.cuda.synchronize()
        sgl.sgl_check(ws)
        assert torch.equal(o, o0) and torch.equal(lse, l0)
        Oref, Lref = decode_attention(case.oracle_q(), W.RowView(case.K), W.RowView(case.V), case.oracle_table,
                                      case.out["seq_lens"])
        assert_close(o.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64), Oref, Lref,
                     *tolerances(case.w))
    finally:
        case.close()


# ---------------------------------------------------------------------------
# FP8 (E4M3) KV cache
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name,num_sms", [("llama3_8b_decode_small", 0), ("llama3_8b_decode_small", 3),
                                          ("multiturn_small", 0), ("fork_tree_small", 0)])
def test_decode_fp8_kv_elementwise(name, num_sms):
    """FP8 pools (per-tensor scales) against the oracle on the decoded values."""
    from oracle.fp8 import DequantView
    case = Case(name)
    try:
        ks, vs = 1.0 / 32, 1.0 / 48
        k8, v8 = W.quantize_e4m3(case.K, ks), W.quantize_e4m3(case.V, vs)
        w = case.w
        p = sgl.make_params(sgl.SGL_DTYPE_BF16_FP8KV, case.B, w.Hq, w.Hkv, w.d, case.S, w.page_size,
                            num_sms=num_sms, k_scale=ks, v_scale=vs)
        plan = sgl.sgl_decode_plan(p, case.out["seq_lens"], sgl.sgl_groups_view(case.groups))
        ws = torch.zeros(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
        sgl.sgl_plan_upload(plan, ws)
        qd = case.q_host().cuda()
        table = torch.from_numpy(case.out["req_to_token"]).cuda()
        seq = torch.from_numpy(case.out["seq_lens"]).cuda()
        o = torch.empty_like(qd)
        lse = torch.empty(case.B, w.Hq, dtype=torch.float32, device="cuda")
        sgl.sgl_decode_attn(qd, k8.cuda(), v8.cuda(), table, seq, plan, o, lse, ws)
        sgl.sgl_check(ws)
        Oref, Lref = decode_attention(case.oracle_q(), DequantView(k8, ks), DequantView(v8, vs), case.oracle_table,
                                      case.out["seq_lens"])
        assert_close(o.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64), Oref, Lref, *tolerances(w))
        del plan
    finally:
        case.close()


@pytest.mark.parametrize("name", ["llama3_8b_decode", "fork_tree"])
def test_decode_fp8_full_size(name):
    """FP8 pools at the full workload sizes, in the benchmark's launch
    configuration (the device's SM count), on every request."""
    from oracle.fp8 import DequantView
    case = Case(name)
    try:
        ks, vs = 1.0 / 64, 1.0 / 64
        k8d = W.quantize_e4m3(case.K.cuda(), ks)
        v8d = W.quantize_e4m3(case.V.cuda(), vs)
        w = case.w
        p = sgl.make_params(sgl.SGL_DTYPE_BF16_FP8KV, case.B, w.Hq, w.Hkv, w.d, case.S, w.page_size,
                            k_scale=ks, v_scale=vs)
        plan = sgl.sgl_decode_plan(p, case.out["seq_lens"], sgl.sgl_groups_view(case.groups))
        assert sgl.sgl_plan_info(plan)["num_wide_items"] > 0
        ws = torch.zeros(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
        sgl.sgl_plan_upload(plan, ws)
        qd = case.q_host().cuda()
        table = torch.from_numpy(case.out["req_to_token"]).cuda()
        seq = torch.from_numpy(case.out["seq_lens"]).cuda()
        o = torch.empty_like(qd)
        lse = torch.empty(case.B, w.Hq, dtype=torch.float32, device="cuda")
        sgl.sgl_decode_attn(qd, k8d, v8d, table, seq, plan, o, lse, ws)
        sgl.sgl_check(ws)
        Oref, Lref = decode_attention(case.oracle_q(), DequantView(k8d.cpu(), ks), DequantView(v8d.cpu(), vs),
                                      case.oracle_table, case.out["seq_lens"])
        do, dl = assert_close(o.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64), Oref, Lref,
                              *tolerances(w))
        print("%s fp8: O max-abs %.3g, LSE max-abs %.3g" % (name, do, dl))
        del plan
    finally:
        case.close()


@pytest.mark.parametrize("name", ["llama3_8b_decode_small", "multiturn_small"])
def test_decode_fp8_subnormal_codes(name):
    """Every K and V code an E4M3 subnormal (exponent field 0: values m 2^-9,
    m < 8), with scales 2^6 so that they matter: the conversions must keep
    them exact on both the tile and the streaming paths (a flush to zero
    would zero every score)."""
    from oracle.fp8 import DequantView
    case = Case(name)
    try:
        ks = vs = 64.0
        k8 = W.quantize_e4m3(case.K, 1.0) & 0x87
        v8 = W.quantize_e4m3(case.V, 1.0) & 0x87
        assert int((k8 & 0x78).max()) == 0 and int((k8 & 0x07).max()) == 7
        w = case.w
        p = sgl.make_params(sgl.SGL_DTYPE_BF16_FP8KV, case.B, w.Hq, w.Hkv, w.d, case.S, w.page_size,
                            k_scale=ks, v_scale=vs)
        plan = sgl.sgl_decode_plan(p, case.out["seq_lens"], sgl.sgl_groups_view(case.groups))
        if name.startswith("llama3"):
            assert sgl.sgl_plan_info(plan)["num_wide_items"] > 0   # the tile path is exercised
        ws = torch.zeros(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
        sgl.sgl_plan_upload(plan, ws)
        qd = case.q_host().cuda()
        table = torch.from_numpy(case.out["req_to_token"]).cuda()
        seq = torch.from_numpy(case.out["seq_lens"]).cuda()
        o = torch.empty_like(qd)
        lse = torch.empty(case.B, w.Hq, dtype=torch.float32, device="cuda")
        sgl.sgl_decode_attn(qd, k8.cuda(), v8.cuda(), table, seq, plan, o, lse, ws)
        sgl.sgl_check(ws)
        Oref, Lref = decode_attention(case.oracle_q(), DequantView(k8, ks), DequantView(v8, vs), case.oracle_table,
                                      case.out["seq_lens"])
        assert_close(o.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64), Oref, Lref, *tolerances(w))
        del plan
    finally:
        case.close()


def _fp8_extend(case, ks, vs):
    pre = case.out["prefix_lens"]
    ext = case.out["seq_lens"] - pre
    w = case.w
    k8, v8 = W.quantize_e4m3(case.K.cuda(), ks), W.quantize_e4m3(case.V.cuda(), vs)
    p = sgl.make_params(sgl.SGL_DTYPE_BF16_FP8KV, case.B, w.Hq, w.Hkv, w.d, case.S, w.page_size, k_scale=ks,
                        v_scale=vs, host_prefix_lens=pre, host_extend_lens=ext)
    ws = torch.zeros(sgl.sgl_extend_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    qd = case.q_host().cuda()
    o = torch.empty_like(qd)
    lse = torch.empty(qd.shape[0], w.Hq, dtype=torch.float32, device="cuda")
    sgl.sgl_extend_attn(qd, k8, v8, torch.from_numpy(case.out["req_to_token"]).cuda(), torch.from_numpy(pre).cuda(),
                        torch.from_numpy(ext).cuda(), p, o, lse, ws)
    sgl.sgl_check(ws)
    return o.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64), k8.cpu(), v8.cpu(), pre, ext, p


@pytest.mark.parametrize("name", ["extend_small", "extend"])
def test_extend_fp8_kv(name):
    """Extend (cached prefix + causal new block) over FP8 pools against the
    oracle on the decoded values: every row at test size; at the full size
    every row of request 2 and sampled rows of the others."""
    from oracle.attention import extend_attention
    from oracle.fp8 import DequantView
    case = Case(name)
    try:
        ks, vs = 1.0 / 64, 1.0 / 48
        O, L, k8, v8, pre, ext, p = _fp8_extend(case, ks, vs)
        rows = None
        if name == "extend":
            rows = full_and_sampled_rows(ext, (2,), 2, (127, 128))
        Oref, Lref = extend_attention(case.oracle_q(), DequantView(k8, ks), DequantView(v8, vs), case.oracle_table,
                                      pre, ext, rows=rows)
        do, dl = assert_close(O, L, Oref, Lref, *tolerances(case.w), rows=rows)
        print("%s fp8 extend: O max-abs %.3g, LSE max-abs %.3g" % (name, do, dl))
    finally:
        case.close()


@pytest.mark.parametrize("name", ["extend_small", "extend"])
def test_fp8_kv_fused_kv_write(name):
    """The fused KV write into FP8 pools: afterwards the pool holds, bit for
    bit, the oracle's E4M3 codes of each new row / scale at its slot (every
    other slot untouched), and the result equals the oracle's extend over the
    written pool (at the full size: every row of request 2, sampled rows of
    the others)."""
    from oracle.attention import extend_attention
    from oracle.fp8 import DequantView, kv_write_e4m3
    case = Case(name)
    try:
        w = case.w
        pre = case.out["prefix_lens"]
        ext = case.out["seq_lens"] - pre
        ks, vs = 1.0 / 64, 1.0 / 48
        k8, v8 = W.quantize_e4m3(case.K, ks), W.quantize_e4m3(case.V, vs)
        kf, vf = W.make_new_kv(w, int(ext.sum()))
        kn, vn = W.to_dtype(w, kf), W.to_dtype(w, vf)
        kd, vd = k8.cuda(), v8.cuda()
        p = sgl.make_params(sgl.SGL_DTYPE_BF16_FP8KV, case.B, w.Hq, w.Hkv, w.d, case.S, w.page_size, k_scale=ks,
                            v_scale=vs, host_prefix_lens=pre, host_extend_lens=ext)
        ws = torch.zeros(sgl.sgl_extend_workspace_bytes(p), dtype=torch.uint8, device="cuda")
        qd = case.q_host().cuda()
        o = torch.empty_like(qd)
        lse = torch.empty(qd.shape[0], w.Hq, dtype=torch.float32, device="cuda")
        sgl.sgl_extend_attn_kvwrite(qd, kn.cuda(), vn.cuda(), kd, vd, torch.from_numpy(case.out["req_to_token"]).cuda(),
                                    torch.from_numpy(pre).cuda(), torch.from_numpy(ext).cuda(), p, o, lse, ws)
        sgl.sgl_check(ws)
        Kexp, Vexp = kv_write_e4m3(k8.numpy().copy(), v8.numpy().copy(), kn.float().numpy(), vn.float().numpy(), ks,
                                   vs, case.oracle_table, pre, ext)
        assert np.array_equal(kd.cpu().numpy(), Kexp) and np.array_equal(vd.cpu().numpy(), Vexp)
        rows = full_and_sampled_rows(ext, (2,), 4, (127, 128)) if name == "extend" else None
        Oref, Lref = extend_attention(case.oracle_q(), DequantView(torch.from_numpy(Kexp), ks),
                                      DequantView(torch.from_numpy(Vexp), vs), case.oracle_table, pre, ext, rows=rows)
        do, dl = assert_close(o.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64), Oref, Lref,
                              *tolerances(w), rows=rows)
        print("%s fp8 fused write: O max-abs %.3g, LSE max-abs %.3g" % (name, do, dl))
    finally:
        case.close()


def test_fp8_query_outside_f16_is_reported():
    """With FP8 pools the query enters the MMAs as f16: an element of
    magnitude 2^16 or more (no f16 value) is reported by sgl_check as
    SGL_ERR_BOUNDS -- on the tile path and the streaming path of decode and
    in extend -- while the same call with the element in range is clean."""
    from tests._harness import run_extend
    ks = vs = 1.0 / 64
    case = Case("llama3_8b_decode_small")
    try:
        w = case.w
        k8, v8 = W.quantize_e4m3(case.K, ks).cuda(), W.quantize_e4m3(case.V, vs).cuda()
        p = sgl.make_params(sgl.SGL_DTYPE_BF16_FP8KV, case.B, w.Hq, w.Hkv, w.d, case.S, w.page_size, k_scale=ks,
                            v_scale=vs)
        plan = sgl.sgl_decode_plan(p, case.out["seq_lens"], sgl.sgl_groups_view(case.groups))
        assert sgl.sgl_plan_info(plan)["num_wide_items"] > 0   # request 0 is on a tile and on a stream
        ws = torch.zeros(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
        sgl.sgl_plan_upload(plan, ws)
        table = torch.from_numpy(case.out["req_to_token"]).cuda()
        seq = torch.from_numpy(case.out["seq_lens"]).cuda()
        for big, expect in ((65280.0, None), (65536.0, -5), (-1e6, -5)):
            qd = case.q_host().clone()
            qd[0, 0, 5] = big
            qd = qd.cuda()
            o = torch.empty_like(qd)
            lse = torch.empty(case.B, w.Hq, dtype=torch.float32, device="cuda")
            sgl.sgl_decode_attn(qd, k8, v8, table, seq, plan, o, lse, ws)
            if expect is None:
                sgl.sgl_check(ws)
            else:
                with pytest.raises(sgl.SglError) as e:
                    sgl.sgl_check(ws)
                assert e.value.status == expect
        del plan
    finally:
        case.close()
    case = Case("extend_small")
    try:
        big_q = case.q_host().clone()
        big_q[3, 1, 7] = 1e5
        case.b.q = big_q.float().numpy()
        with pytest.raises(sgl.SglError) as e:
            _fp8_extend(case, ks, vs)
        assert e.value.status == -5
    finally:
        case.close()


@pytest.mark.parametrize("name,steps", [("llama3_8b_decode_small", 1), ("llama3_8b_decode_small", 9),
                                        ("fork_tree_small", 40), ("multiturn_small", 23), ("tiny_fp32", 5)])
def test_plan_reused_after_decode_steps(name, steps):
    """A plan made for a batch stays valid after every request has grown by
    `steps` tokens (sgl_batch_append): the requests' trailing pieces read up
    to the grown seq_lens.  The batch adds a copy of request 0 (its context
    ends in a shared segment) and an empty request; the result equals the
    oracle on the grown batch, whose table the oracle builds with its own
    append_step."""
    from oracle.tree import append_step
    w = W.get(name)
    base = W.make_batch(w, 0).all_tokens()
    seqs = list(base) + [list(base[0]), []]
    rng = np.random.default_rng(31 + steps)
    q = rng.standard_normal((len(seqs), w.Hq, w.d), dtype=np.float32)
    case = Case(None, workload=w, seqs=seqs, q=q)
    try:
        B = case.B
        ld = case.out["req_to_token"].shape[1] + steps
        tab = np.full((B, ld), -1, dtype=np.int32)
        tab[:, :ld - steps] = case.out["req_to_token"]
        seq = case.out["seq_lens"].copy()
        p = case.params()
        plan = sgl.sgl_decode_plan(p, seq, sgl.sgl_groups_view(case.groups))
        ws = torch.zeros(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
        sgl.sgl_plan_upload(plan, ws)
        rows = [list(case.oracle_table[r, :seq[r]]) for r in range(B)]
        for _ in range(steps):
            sgl.sgl_batch_append(case.tree, tab, seq, None)
            append_step(case.trie, rows)
        oracle_table = np.full((B, ld), -1, dtype=np.int64)
        for r, row in enumerate(rows):
            oracle_table[r, :len(row)] = row
        kd, vd = case.device_pool()
        qd = case.q_host().cuda()
        o = torch.empty_like(qd)
        lse = torch.empty(B, w.Hq, dtype=torch.float32, device="cuda")
        sgl.sgl_decode_attn(qd, kd, vd, torch.from_numpy(tab).cuda(), torch.from_numpy(seq).cuda(), plan, o, lse, ws)
        sgl.sgl_check(ws)
        Oref, Lref = decode_attention(case.oracle_q(), W.RowView(case.K), W.RowView(case.V), oracle_table,
                                      np.array([len(r) for r in rows]))
        assert_close(o.double().cpu().numpy(), lse.cpu().numpy().astype(np.float64), Oref, Lref, *tolerances(w))
    finally:
        case.close()


def test_reused_plan_reports_a_batch_that_shrank():
    """A request shorter than its planned trailing piece start sets error bit
    1 (SGL_ERR_BOUNDS from sgl_check) instead of reading stale positions."""
    case = Case("llama3_8b_decode_small")
    try:
        p = case.params()
        seq = case.out["seq_lens"].copy()
        plan = sgl.sgl_decode_plan(p, seq, sgl.sgl_groups_view(case.groups))
        ws = torch.zeros(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
        sgl.sgl_plan_upload(plan, ws)
        kd, vd = case.device_pool()
        qd = case.q_host().cuda()
        o = torch.empty_like(qd)
        lse = torch.empty(case.B, case.w.Hq, dtype=torch.float32, device="cuda")
        short = seq.copy()
        short[0] = 1   # request 0 shrank below its planned pieces
        sgl.sgl_decode_attn(qd, kd, vd, torch.from_numpy(case.out["req_to_token"]).cuda(),
                            torch.from_numpy(short).cuda(), plan, o, lse, ws)
        with pytest.raises(sgl.SglError) as e:
            sgl.sgl_check(ws)
        assert e.value.status == -5
    finally:
        case.close()


def _packed(case):
    """A step's inputs in one pinned host buffer [q | req_to_token | seq_lens]
    and its outputs [O | LSE], with device staging tensors of the same
    layout and views into them."""
    q = case.q_host()
    table = np.ascontiguousarray(case.out["req_to_token"], dtype=np.int32)
    seq = np.ascontiguousarray(case.out["seq_lens"], dtype=np.int32)
    qb, tb, sb = q.numel() * q.element_size(), table.nbytes, seq.nbytes
    ob, lb = qb, case.B * case.w.Hq * 4
    hin = torch.empty(qb + tb + sb, dtype=torch.uint8).pin_memory()
    hin[:qb].copy_(q.reshape(-1).view(torch.uint8))
    hin[qb:qb + tb].copy_(torch.from_numpy(table).reshape(-1).view(torch.uint8))
    hin[qb + tb:].copy_(torch.from_numpy(seq).view(torch.uint8))
    din = torch.empty_like(hin, device="cuda")
    hout = torch.full((ob + lb,), 0xAB, dtype=torch.uint8).pin_memory()
    dout = torch.empty_like(hout, device="cuda")
    views = dict(q=din[:qb].view(q.dtype).view(q.shape), table=din[qb:qb + tb].view(torch.int32).view(table.shape),
                 seq=din[qb + tb:].view(torch.int32), o=dout[:ob].view(q.dtype).view(q.shape),
                 lse=dout[ob:].view(torch.float32).view(case.B, case.w.Hq))
    return hin, din, hout, dout, views, ob


@pytest.mark.parametrize("name", ["llama3_8b_decode_small", "tiny_fp32"])
def test_decode_step_from_host_memory(name):
    """sgl_decode_step (input copy, decode, output copy in one call) gives the
    same bytes as the copies and sgl_decode_attn made separately, and the
    oracle's result."""
    case = Case(name)
    try:
        kd, vd = case.device_pool()
        plan = sgl.sgl_decode_plan(case.params(), case.out["seq_lens"], sgl.sgl_groups_view(case.groups))
        ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
        sgl.sgl_plan_upload(plan, ws)
        hin, din, hout, dout, v, ob = _packed(case)
        sgl.sgl_decode_step(hin, din, v["q"], kd, vd, v["table"], v["seq"], plan, v["o"], v["lse"], dout, hout, ws)
        torch.cuda.synchronize()
        sgl.sgl_check(ws)
        o_ref = torch.empty_like(v["o"])
        lse_ref = torch.empty_like(v["lse"])
        sgl.sgl_decode_attn(v["q"], kd, vd, v["table"], v["seq"], plan, o_ref, lse_ref, ws)
        torch.cuda.synchronize()
        assert torch.equal(hout[:ob], o_ref.reshape(-1).view(torch.uint8).cpu())
        assert torch.equal(hout[ob:], lse_ref.reshape(-1).view(torch.uint8).cpu())
        O = hout[:ob].view(v["o"].dtype).view(v["o"].shape).double().numpy()
        L = hout[ob:].view(torch.float32).view(case.B, case.w.Hq).double().numpy()
        Oref, Lref = decode_attention(case.oracle_q(), W.RowView(case.K), W.RowView(case.V), case.oracle_table,
                                      case.out["seq_lens"])
        assert_close(O, L, Oref, Lref, *tolerances(case.w))
    finally:
        case.close()


def test_decode_step_refuses_before_any_copy():
    """A refused step queues nothing: the host output buffer keeps its bytes."""
    case = Case("llama3_8b_decode_small")
    try:
        kd, vd = case.device_pool()
        plan = sgl.sgl_decode_plan(case.params(), case.out["seq_lens"], sgl.sgl_groups_view(case.groups))
        hin, din, hout, dout, v, ob = _packed(case)
        small = torch.zeros(256, dtype=torch.uint8, device="cuda")   # below the plan's workspace
        with pytest.raises(sgl.SglError) as e:
            sgl.sgl_decode_step(hin, din, v["q"], kd, vd, v["table"], v["seq"], plan, v["o"], v["lse"], dout, hout,
                                small)
        assert e.value.status == -7
        torch.cuda.synchronize()
        assert bool((hout == 0xAB).all())
    finally:
        case.close()
