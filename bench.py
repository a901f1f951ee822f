#!/usr/bin/env python
"""Benchmark of the RadixAttention hot path on GB300.

One step = one decode batch of the Llama-3-8B-shaped workload (64 requests
sharing a 2048-token system prefix, suffixes 64..512 tokens, Hq 32 / Hkv 8 /
d 128, bf16, 2^20-slot pool, random slots): prefix-group planning is done
once per batch instance, and the timed step is the decode call (split-KV
partial + log-sum-exp merge) through the C ABI.  The metric is unique-KV
GB/s: the K/V bytes of every prefix-group segment counted once per step.

  * Device value: K steps replayed from CUDA graphs, rotating over batch
    instances whose combined unique KV is several times the 129 MB L2, CUDA
    events around the K steps, max over ranks.
  * e2e: the same metric through the public API from host buffers on one
    growing batch -- the batch built from the tree, then per step one new
    slot per request (table and prefix groups grown), planning, plan upload,
    pinned H2D of q and the tables, the decode call, D2H of O and LSE, and
    at the end the sequences cached in the tree -- wall clock per step, the
    host preparing step s+1 while the GPU runs step s.
  * extend: TFLOP/s of the chunked-prefill workload (8 requests, cached
    4096-token prefix + 512 causal new tokens, Hq 64 / Hkv 8), unmasked
    query-key pairs x 4 d FLOP.
  * roofline: the decode call (the persistent partial kernel + the merge
    kernel); achieved = unique-KV bytes per call / call time, against the
    measured HBM copy bandwidth; ncu DRAM traffic per call from profiles/
    when current.
  * cpu_baseline / --impl reference: the float64 oracle (test
    infrastructure) timed on host cores on a bounded sample of the workload.

Multi-GPU: the path has no exchange step; each rank runs an independent
replica (weak scaling), value = bytes of all ranks / max time.
"""

import argparse
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "decode attn unique-KV GB/s (% of HBM peak); extend attn TFLOP/s; tokens/s"
DECODE_WORKLOAD = "llama3_8b_decode"
EXTEND_WORKLOAD = "extend"
L2_BYTES = 129 * 1000 * 1000


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--instances", type=int, default=8)
    ap.add_argument("--graph-len", type=int, default=400)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--extend-steps", type=int, default=20)
    ap.add_argument("--no-extend", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget-s", type=float, default=60.0)
    ap.add_argument("--num-sms", type=int, default=0, help="decode planning target (0: the device's SM count)")
    ap.add_argument("--workload", default="",
                    help="time only this decode workload (fork_tree, multiturn, multiturn_noshare, tiny_fp32; "
                         "profiling), with --instances instances and --steps calls")
    ap.add_argument("--only", choices=["all", "decode", "extend", "mla"], default="all",
                    help="decode: skip the extend line; extend: time only the extend workload (profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sched", action="store_true", help="skip the host scheduling simulation")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8 KV decode object")
    ap.add_argument("--no-mla", action="store_true", help="skip the MLA decode object")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the fork_tree / multiturn / multiturn_noshare / tiny_fp32 objects")
    ap.add_argument("--pool-slots", type=int, default=0,
                    help="decode pool size override (0: the workload's 2^20 slots); small pools serve ncu captures")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def job_timing(ms_local, bytes_per_rank, world, device):
    """(max over the ranks of the timed region in ms, whole-job GB/s): every
    rank processed bytes_per_rank in its timed region (independent replicas,
    weak scaling).  `device` holds the reduction tensor (cuda under NCCL, cpu
    under gloo)."""
    import torch
    ms_t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(ms_t, op=torch.distributed.ReduceOp.MAX)
    ms_max = float(ms_t.item())
    return ms_max, bytes_per_rank * world / (ms_max / 1e3) / 1e9


def kv_bytes_per_token(w):
    return 2 * w.Hkv * w.d * (4 if w.dtype == "f32" else 2)


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        self.t_start = time.time()

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1].split()[0]))
                mx = float(f[2].split()[0])
            except ValueError:
                continue
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- reference arm (oracle)
def reference_arm(args, budget_s, steps, warmup):
    """Time the float64 oracle (shared-aware decode) on bounded samples of the workload."""
    import numpy as np
    import workloads as W
    from oracle.attention import decode_attention, decode_attention_shared
    from oracle.groups import prefix_groups
    from oracle.tree import RadixTrie, build_batch

    w = W.get(DECODE_WORKLOAD)
    b = W.make_batch(w, 0)
    order, K, V = W.make_pool(w)
    Kv, Vv = W.RowView(K), W.RowView(V)
    trie = RadixTrie(K.shape[0], w.page_size, order)
    seqs = b.all_tokens()
    rows, _, _ = build_batch(trie, seqs)
    q = W.to_dtype(w, b.q).double().numpy()
    per_tok = kv_bytes_per_token(w)

    def sample(m):
        sub = rows[:m]
        ld = max(len(r) for r in sub)
        t = np.full((m, ld), -1, dtype=np.int64)
        for i, r in enumerate(sub):
            t[i, :len(r)] = r
        lens = np.array([len(r) for r in sub])
        g = prefix_groups(t, lens)
        ub = sum(int(e) - int(s) for s, e in zip(g["seg_begin"], g["seg_end"])) * per_tok
        return t, lens, g, ub

    # calibrate the per-step sample so warmup + steps fit the budget
    t1, l1, g1, _ = sample(1)
    c0 = time.perf_counter()
    decode_attention_shared(q[:1], Kv, Vv, t1, l1, g1)
    one = time.perf_counter() - c0
    per_step = budget_s / max(1, steps + warmup)
    m = int(max(1, min(len(rows), per_step / max(one, 1e-6))))
    t, lens, g, ub = sample(m)
    for _ in range(warmup):
        decode_attention_shared(q[:m], Kv, Vv, t, lens, g)
    c0 = time.perf_counter()
    for _ in range(steps):
        decode_attention_shared(q[:m], Kv, Vv, t, lens, g)
    el = time.perf_counter() - c0
    c1 = time.perf_counter()
    decode_attention(q[:m], Kv, Vv, t, lens)
    unshared_s = time.perf_counter() - c1
    gbs = ub * steps / el / 1e9
    return {
        "value": gbs, "seconds_per_step": el / steps, "requests": m, "unique_bytes": ub,
        "unshared_seconds_per_step": unshared_s,
        "sample": "%d of %d requests of batch instance 0 (%d unique KV tokens), shared-aware float64 decode, "
                  "%d steps" % (m, len(rows), ub // per_tok, steps),
    }


def host_cores():
    """The host cores this process may run on."""
    return len(os.sched_getaffinity(0))


def set_blas_threads():
    """BLAS threads = the host cores (before numpy is first imported); the
    oracle's own loop over requests and heads stays one Python thread."""
    n = str(host_cores())
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = n
    return int(n)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    cores = set_blas_threads()
    r = reference_arm(args, args.ref_budget_s, max(1, args.steps), max(0, min(args.warmup, 3)))
    line = {
        "metric": METRIC, "value": r["value"], "unit": "GB/s", "impl": "reference", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["seconds_per_step"] * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": DECODE_WORKLOAD, "batch": 64, "prefix": 2048, "suffix": "U[64,512]",
                   "heads": "Hq32/Hkv8/d128", "pool_slots": 1 << 20, "sample_requests": r["requests"]},
        "cpu_baseline": {"value": r["value"], "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": r["sample"] + "; BLAS threads %d, the oracle's loop one Python thread" % cores,
                         "seconds_per_step": r["seconds_per_step"],
                         "unshared_seconds_per_step": r["unshared_seconds_per_step"]},
        "e2e": {"value": r["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline_subprocess(budget_s=15.0):
    n = str(host_cores())
    env = dict(os.environ, OMP_NUM_THREADS=n, OPENBLAS_NUM_THREADS=n, MKL_NUM_THREADS=n, RANK="0", WORLD_SIZE="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--steps", "3", "--warmup", "1",
           "--ref-budget-s", str(budget_s)]
    try:
        out = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
        for l in out.stdout.splitlines()[::-1]:
            if l.startswith("{"):
                d = json.loads(l)
                return dict(d["cpu_baseline"])
    except Exception as e:  # the baseline is context only
        return {"value": None, "unit": "GB/s", "cores": host_cores(), "kind": "oracle", "sample": "failed: %s" % e}
    return {"value": None, "unit": "GB/s", "cores": host_cores(), "kind": "oracle", "sample": "no output"}


# --------------------------------------------------------------------------- native arm
def setup_decode(sgl, W, torch, n_inst, num_sms=0, pool_slots=0, name=DECODE_WORKLOAD):
    import dataclasses
    w = W.get(name)
    if pool_slots:
        w = dataclasses.replace(w, num_slots=int(pool_slots))
    S = W.pool_slots(w, n_inst)
    order, K, V = W.make_pool(w, num_slots=S)
    kd, vd = K.cuda(), V.cuda()
    del K, V
    tree = sgl.sgl_tree_create(S, w.page_size, order)
    per_tok = kv_bytes_per_token(w)
    dt = sgl.SGL_DTYPE_F32 if w.dtype == "f32" else sgl.SGL_DTYPE_BF16
    inst = []
    for i in range(n_inst):
        b = W.make_batch(w, i)
        seqs = b.all_tokens()
        groups = sgl.sgl_groups_create()
        out = sgl.sgl_build_batch(tree, seqs, groups=groups)
        view = sgl.sgl_groups_view(groups)
        gnp = sgl.groups_as_numpy(view)
        ub = int((gnp["seg_end"] - gnp["seg_begin"]).sum()) * per_tok
        p = sgl.make_params(dt, len(seqs), w.Hq, w.Hkv, w.d, S, w.page_size, num_sms=num_sms)
        plan = sgl.sgl_decode_plan(p, out["seq_lens"], view)
        ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
        sgl.sgl_plan_upload(plan, ws)
        q = W.to_dtype(w, b.q).cuda()
        inst.append(dict(seqs=seqs, groups=groups, out=out, plan=plan, ws=ws, q=q,
                         table=torch.from_numpy(out["req_to_token"]).cuda(),
                         seq=torch.from_numpy(out["seq_lens"]).cuda(),
                         o=torch.empty_like(q), lse=torch.empty(len(seqs), w.Hq, dtype=torch.float32, device="cuda"),
                         ub=ub, unshared=int(out["seq_lens"].sum()) * per_tok, B=len(seqs)))
        for r in range(len(seqs)):   # the batch's requests release their references; the cache keeps the KV
            sgl.sgl_tree_finish(tree, int(out["last_nodes"][r]), out["req_to_token"][r], len(seqs[r]))
    torch.cuda.synchronize()
    return w, tree, kd, vd, inst


def graph_time(torch, fn, calls, n):
    """ms per call of n back-to-back calls fn(calls[j % len(calls)]) captured
    in one CUDA graph (replayed once to warm, then timed with CUDA events on
    the current stream)."""
    n = max(len(calls), n - n % len(calls))
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            for j in range(n):
                fn(calls[j % len(calls)])
    torch.cuda.current_stream().wait_stream(st)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n, n


def bench_decode_workload(sgl, W, torch, name, n_inst, n_calls, hbm_peak, num_sms=0, fp8=False):
    """Another decode workload timed like the headline: one CUDA graph of
    back-to-back calls rotating over n_inst batch instances, CUDA events.
    Returns unique-KV bytes per call, GB/s and fractions of the measured HBM
    copy peak and of 8 TB/s; with fp8, the same batches on an E4M3 copy of
    the pool too."""
    w, tree, kd, vd, inst = setup_decode(sgl, W, torch, n_inst, num_sms, name=name)
    for s in range(max(3, len(inst))):
        decode_call(sgl, kd, vd, inst[s % len(inst)])
    torch.cuda.synchronize()
    for it in inst:
        sgl.sgl_check(it["ws"])
    ms, n = graph_time(torch, lambda it: decode_call(sgl, kd, vd, it), inst, n_calls)
    for it in inst:
        sgl.sgl_check(it["ws"])
    ub = sum(it["ub"] for it in inst) / len(inst)
    uns = sum(it["unshared"] for it in inst) / len(inst)
    gbs = ub / (ms / 1e3) / 1e9
    info = sgl.sgl_plan_info(inst[0]["plan"])
    r = {"workload": name, "batch": inst[0]["B"], "heads": "Hq%d/Hkv%d/d%d" % (w.Hq, w.Hkv, w.d), "dtype": w.dtype,
         "page_size": w.page_size, "pool_slots": kd.shape[0], "instances": len(inst),
         "unique_kv_bytes_per_call": int(ub), "unshared_kv_bytes_per_call": int(uns),
         "us_per_call": ms * 1e3, "unique_kv_gbs": gbs, "frac_of_hbm": gbs / hbm_peak, "frac_of_8TBs": gbs / 8000.0,
         "tokens_per_s": inst[0]["B"] / (ms / 1e3), "calls_timed": n,
         "wide_items": info["num_wide_items"], "items": info["num_items"],
         "l2": "%d instance(s), %.0f MB unique KV in all (L2 %d MB)" % (len(inst), ub * len(inst) / 1e6,
                                                                       L2_BYTES // 1000000)}
    if fp8:
        r["fp8_kv"] = bench_fp8(sgl, W, torch, w, kd, vd, inst, n_calls, hbm_peak, num_sms, name=name)
        r["fp8_kv"]["speedup_vs_bf16"] = ms / r["fp8_kv"]["ms_per_call"]
    del inst
    sgl.sgl_tree_destroy(tree)
    del kd, vd
    torch.cuda.empty_cache()
    return r


def decode_call(sgl, kd, vd, it):
    sgl.sgl_decode_attn(it["q"], kd, vd, it["table"], it["seq"], it["plan"], it["o"], it["lse"], it["ws"])


REPLAN = 32   # e2e: decode steps between plans


def e2e_decode(sgl, W, torch, w, tree, kd, vd, inst, steps, num_sms=0):
    """Decode steps of a serving loop through the public API from host
    buffers, on one batch that grows, with the host one step ahead of the
    GPU (the overlap scheduling of the CS349D lecture-16 notes §2.2: while
    the GPU runs step s, the CPU prepares all of step s+1's metadata).
    Step 0 runs sgl_build_batch (match; allocate and insert the unmatched
    tail; emit the prefix groups; the slot table goes straight into the
    pinned staging buffer); every later step's metadata is sgl_batch_append
    (one new slot per request, the table and prefix groups grown; the tree
    untouched).  A plan is reused while the requests grow (its trailing
    pieces read up to the run-time lengths) and rebuilt every REPLAN steps
    (sgl_decode_plan, then sgl_plan_upload into the other of two workspaces,
    while the GPU runs the step before).  Each step is one sgl_decode_step
    call: its inputs (Q, the slot table, the lengths: one pinned buffer laid
    out like one device buffer) to the device in one copy, the decode, O and
    LSE back in one copy; the loop then waits for them.  After the last step
    sgl_tree_cache_finished_batch caches every sequence.  All of it is
    timed.  The per-step GPU calls go straight to the C ABI with the
    buffers' addresses taken once (as a C or C++ serving loop would call
    it).  The table needs no second staging buffer: an append only writes
    positions past every row's length in the step in flight, which that
    step never reads; the lengths are copied into the staging buffer when
    their step is launched.  Returns (GB/s of unique KV, h2d bytes/step,
    d2h bytes/step, s/step, host us per stage, build and finish amortised
    over the steps)."""
    import ctypes
    import numpy as np
    lib = sgl._lib()
    S = kd.shape[0]
    it = inst[0]
    B = it["B"]
    lens0 = np.array([len(t) for t in it["seqs"]], dtype=np.int64)
    cap = int(lens0.max()) + steps
    toks = np.zeros((B, cap), dtype=np.int32)
    for r, t in enumerate(it["seqs"]):
        toks[r, :len(t)] = t
    rng = np.random.default_rng(12)
    toks_new = rng.integers(0, W.VOCAB, size=(steps, B)).astype(np.int32)
    ld = cap
    # inputs [q | req_to_token | seq_lens], outputs [O | LSE], each one
    # pinned host buffer and one device buffer of the same layout
    qb, tb, sb = it["q"].numel() * 2, B * ld * 4, B * 4
    ob, lb = it["o"].numel() * 2, it["lse"].numel() * 4
    hin = torch.empty(qb + tb + sb, dtype=torch.uint8).pin_memory()
    din = torch.empty(qb + tb + sb, dtype=torch.uint8, device="cuda")
    hout = torch.empty(ob + lb, dtype=torch.uint8).pin_memory()
    dout = torch.empty(ob + lb, dtype=torch.uint8, device="cuda")
    hin[:qb].view(torch.bfloat16).copy_(it["q"].cpu().reshape(-1).view(torch.bfloat16))
    tab_np = hin[qb:qb + tb].view(torch.int32).view(B, ld).numpy()
    hseq_np = hin[qb + tb:].view(torch.int32).numpy()
    seq_np = np.zeros(B, dtype=np.int32)   # the lengths the host side works on
    groups = sgl.sgl_groups_create()
    # the largest plan of the run sizes the workspaces (allocated before timing)
    wsz = 4 * it["plan"].workspace_bytes + (1 << 20)
    ws = [torch.zeros(wsz, dtype=torch.uint8, device="cuda") for _ in range(2)]
    vp = ctypes.c_void_p
    base_in, base_out = din.data_ptr(), dout.data_ptr()
    args_fixed = dict(q=vp(base_in), k=vp(kd.data_ptr()), v=vp(vd.data_ptr()), tab=vp(base_in + qb),
                      seq=vp(base_in + qb + tb), o=vp(base_out), lse=vp(base_out + ob))
    ws_ptr = [vp(x.data_ptr()) for x in ws]
    hin_p, hout_p = vp(hin.data_ptr()), vp(hout.data_ptr())
    nin, nout = qb + tb + sb, ob + lb
    stream = vp(torch.cuda.current_stream().cuda_stream)
    per_tok = kv_bytes_per_token(w)
    ub0 = it["ub"]
    rows = np.arange(B)
    stage = dict(build=0.0, append=0.0, plan=0.0, upload=0.0, launch=0.0, wait=0.0, finish=0.0)
    done = torch.cuda.Event()
    total_b = 0

    def plan_step():
        c1 = time.perf_counter()
        p = sgl.make_params(sgl.SGL_DTYPE_BF16, B, w.Hq, w.Hkv, w.d, S, w.page_size, num_sms=num_sms)
        pl = sgl.sgl_decode_plan(p, seq_np, sgl.sgl_groups_view(groups))
        if pl.workspace_bytes > wsz:
            raise RuntimeError("e2e workspace too small")
        stage["plan"] += time.perf_counter() - c1
        return pl

    def upload(pl, k):
        c1 = time.perf_counter()
        st = lib.sgl_plan_upload(pl.handle, ws_ptr[k], wsz, stream)
        if st:
            raise sgl.SglError(st, "sgl_plan_upload")
        stage["upload"] += time.perf_counter() - c1

    torch.cuda.synchronize()
    t0 = time.perf_counter()
    c0 = time.perf_counter()
    out = sgl.sgl_build_batch(tree, toks, groups=groups, req_to_token=tab_np, seq_lens=seq_np, lens=lens0)
    stage["build"] += time.perf_counter() - c0
    plan = plan_step()
    upload(plan, 0)
    up_bytes = sgl.sgl_plan_info(plan)["upload_bytes"]
    d2h = ob + lb
    a = args_fixed
    cur = 0   # the workspace of the plan in use
    for s in range(steps):
        c0 = time.perf_counter()
        hseq_np[:] = seq_np
        st = lib.sgl_decode_step(hin_p, a["q"], nin, a["q"], a["k"], a["v"], a["tab"], ld, a["seq"], plan.handle,
                                 a["o"], a["lse"], a["o"], hout_p, nout, ws_ptr[cur], wsz, stream)
        if st:
            raise sgl.SglError(st, "sgl_decode_step")
        done.record()
        stage["launch"] += time.perf_counter() - c0
        # the shared prefix is unchanged; every request's own suffix grew by one token a step
        total_b += ub0 + s * B * per_tok
        nxt = None
        if s + 1 < steps:
            # step s+1's metadata while the GPU runs step s
            c0 = time.perf_counter()
            sgl.sgl_batch_append(tree, tab_np, seq_np, groups)
            toks[rows, seq_np - 1] = toks_new[s + 1]
            stage["append"] += time.perf_counter() - c0
            if (s + 1) % REPLAN == 0:
                nxt = plan_step()
                upload(nxt, cur ^ 1)
                up_bytes += sgl.sgl_plan_info(nxt)["upload_bytes"]
        c0 = time.perf_counter()
        done.synchronize()   # step s's O and LSE are on the host
        stage["wait"] += time.perf_counter() - c0
        if nxt is not None:
            plan = nxt
            cur ^= 1
    h2d = qb + tb + sb + up_bytes // steps
    c5 = time.perf_counter()
    sgl.sgl_tree_cache_finished_batch(tree, toks, out)
    el = time.perf_counter() - t0
    stage["finish"] += time.perf_counter() - c5
    for x in ws:
        sgl.sgl_check(x)
    sgl.sgl_groups_destroy(groups)
    host_us = {k: v * 1e6 / steps for k, v in stage.items()}
    return total_b / el / 1e9, h2d, d2h, el / steps, host_us


def run_native(args):
    import numpy as np
    import torch
    import radixattention_prefix_shared_radix_gb300 as sgl
    from radixattention_prefix_shared_radix_gb300 import build as sglbuild
    import workloads as W

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    sglbuild.build()
    hbm_peak, bf16_peak, peak_src = peaks()
    if args.only == "mla":
        r = bench_mla(sgl, W, torch, max(4, min(args.steps, 2000)), bf16_peak, hbm_peak, args.num_sms)
        if rank == 0:
            print(json.dumps({"metric": "mla decode ms per call", "value": r["ms_per_call"], "unit": "ms",
                              "n_gpus": world, "mla": r}), flush=True)
        return
    if args.workload:
        r = bench_decode_workload(sgl, W, torch, args.workload, args.instances, max(1, args.steps), hbm_peak,
                                  args.num_sms, fp8=not args.no_fp8)
        if rank == 0:
            print(json.dumps({"metric": "decode us per call", "value": r["us_per_call"], "unit": "us",
                              "n_gpus": world, args.workload: r}), flush=True)
        return
    if args.only == "extend":
        ext = bench_extend(sgl, W, torch, max(3, args.extend_steps), bf16_peak)
        if rank == 0:
            print(json.dumps({"metric": "extend attn TFLOP/s", "value": ext["tflops"], "unit": "TFLOP/s",
                              "n_gpus": world, "extend": ext}), flush=True)
        return

    w, tree, kd, vd, inst = setup_decode(sgl, W, torch, args.instances, args.num_sms, args.pool_slots)
    ub_all = sum(it["ub"] for it in inst)
    warm = max(3, args.warmup)
    for s in range(warm):
        decode_call(sgl, kd, vd, inst[s % len(inst)])
    torch.cuda.synchronize()
    for it in inst:
        sgl.sgl_check(it["ws"])

    # CUDA graphs of back-to-back decode calls rotating over the instances
    K = max(1, args.steps)
    glen = max(1, min(args.graph_len, K))
    glen -= glen % len(inst) if glen >= len(inst) else 0

    def capture(n, start):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for j in range(n):
                    decode_call(sgl, kd, vd, inst[(start + j) % len(inst)])
        torch.cuda.current_stream().wait_stream(s)
        return g

    reps, rem = divmod(K, glen)
    g_main = capture(glen, 0)
    g_rem = capture(rem, 0) if rem else None
    g_main.replay()
    torch.cuda.synchronize()
    bytes_per_step = [inst[j % len(inst)]["ub"] for j in range(glen)]
    total_bytes = sum(bytes_per_step) * reps + sum(bytes_per_step[:rem])

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g_main.replay()
    if g_rem is not None:
        g_rem.replay()
    e1.record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks.stop()
    ms = e0.elapsed_time(e1)
    ms_max, value = job_timing(ms, total_bytes, world, "cuda")
    for it in inst:
        sgl.sgl_check(it["ws"])
    per_call_ms = ms / K
    achieved = (total_bytes / K) / (per_call_ms / 1e3) / 1e9

    # e2e through the public API from host buffers
    e2e_gbs = h2d = d2h = e2e_step_s = e2e_host = None
    if not args.no_e2e:
        e2e_gbs, h2d, d2h, e2e_step_s, e2e_host = e2e_decode(sgl, W, torch, w, tree, kd, vd, inst,
                                                             max(1, min(args.e2e_steps, K)), args.num_sms)

    mla = None
    if not args.no_mla and args.only == "all":
        mla = bench_mla(sgl, W, torch, min(K, 2000), bf16_peak, hbm_peak, args.num_sms)

    fp8 = None
    if not args.no_fp8:
        fp8 = bench_fp8(sgl, W, torch, w, kd, vd, inst, min(K, 2000), hbm_peak, args.num_sms)
        fp8["speedup_vs_bf16"] = per_call_ms / fp8["ms_per_call"]

    others = None
    if not args.no_workloads and args.only == "all":
        # the other decode workloads: parallel-sampling fork tree, multi-turn
        # groups at 80% and 0% sharing (inputs larger than L2 per call), and
        # the tiny fp32 batch (latency only)
        others = {}
        for name, n_inst, n_calls, f8 in (("fork_tree", 4, 400, True), ("multiturn", 1, 100, True),
                                          ("multiturn_noshare", 1, 60, True), ("tiny_fp32", 4, 2000, False)):
            others[name] = bench_decode_workload(sgl, W, torch, name, n_inst, n_calls, hbm_peak, args.num_sms,
                                                 fp8=f8 and not args.no_fp8)

    ext = None
    if not args.no_extend and args.only == "all":
        ext = bench_extend(sgl, W, torch, max(3, args.extend_steps), bf16_peak)

    traffic = profile_traffic("decode_partial")
    launches_per_call = 2   # bf16 decode: the persistent partial kernel and the merge kernel
    B = inst[0]["B"]
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": warm,
        "ms_per_step": ms_max / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": DECODE_WORKLOAD, "batch": B, "prefix": 2048, "suffix": "U[64,512]",
                   "heads": "Hq32/Hkv8/d128", "pool_slots": kd.shape[0], "page_size": 1,
                   "instances": len(inst), "unique_kv_bytes_per_step": ub_all // len(inst),
                   "unshared_kv_bytes_per_step": sum(it["unshared"] for it in inst) // len(inst),
                   "l2": "inputs larger than L2: %d rotating batch instances, %.0f MB unique KV > %d MB L2"
                         % (len(inst), ub_all / 1e6, L2_BYTES // 1000000),
                   "timing": "CUDA graphs of %d back-to-back decode calls, CUDA events" % glen,
                   "parallelism": "replicas" if world > 1 else "single"},
        "tokens_per_s": B * world / (ms_max / 1e3 / K),
        "tokens_per_s_32_layers": B * world / (ms_max / 1e3 / K) / 32,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "peak_source": peak_src,
                     "frac_of_8TBs": achieved / 8000.0, "traffic": traffic,
                     "kernel": "decode call = decode_fused_kernel + decode_merge_kernel (unique-KV bytes / call time)"},
        "e2e": {"value": e2e_gbs, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_step_s * 1e3 if e2e_step_s else None,
                "step": "one growing batch (batch instance 0), the host one step ahead of the GPU: step 0 "
                        "builds it from the tree; while the GPU runs step s the host appends one token per "
                        "request for step s+1 (a slot allocated, the table and prefix groups grown) and, "
                        "every %d steps, plans the batch anew and uploads the plan to a second workspace "
                        "(in between the plan is reused: its trailing pieces read the run-time lengths); "
                        "each step copies Q, the table and the " % REPLAN +
                        "lengths in (one pinned buffer, one copy), decodes and copies O and LSE out (one copy), "
                        "all by one sgl_decode_step call of the C ABI with the buffers' addresses, and waits "
                        "for them; after the last step "
                        "every sequence is cached in the tree and released",
                "host_us_per_step": e2e_host},
        "gpu_launches": K * launches_per_call,
        "clocks": clocks.summary(),
    }
    if fp8 is not None:
        line["fp8_kv"] = fp8
    if mla is not None:
        line["mla"] = mla
    if others is not None:
        line.update(others)
    if ext is not None:
        line["extend"] = ext
    if rank == 0 and args.only == "all" and not args.no_sched:
        line["scheduling"] = bench_scheduling(sgl, W, w)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_subprocess()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def bench_extend(sgl, W, torch, steps, bf16_peak):
    w = W.get(EXTEND_WORKLOAD)
    order, K, V = W.make_pool(w)
    S = K.shape[0]
    kd, vd = K.cuda(), V.cuda()
    b = W.make_batch(w, 0)
    tree = sgl.sgl_tree_create(S, w.page_size, order)
    warm = [b.cached_tokens(r) for r in range(len(b.req_chain))]
    o0 = sgl.sgl_build_batch(tree, warm)
    for r in range(len(warm)):
        sgl.sgl_tree_finish(tree, int(o0["last_nodes"][r]), o0["req_to_token"][r], len(warm[r]))
    seqs = b.all_tokens()
    out = sgl.sgl_build_batch(tree, seqs)
    pre = out["prefix_lens"]
    ext = out["seq_lens"] - pre
    p = sgl.make_params(sgl.SGL_DTYPE_BF16, len(seqs), w.Hq, w.Hkv, w.d, S, w.page_size,
                        host_prefix_lens=pre, host_extend_lens=ext)
    ws = torch.zeros(sgl.sgl_extend_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    q = W.to_dtype(w, b.q).cuda()
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[0], w.Hq, dtype=torch.float32, device="cuda")
    table = torch.from_numpy(out["req_to_token"]).cuda()
    pre_d, ext_d = torch.from_numpy(pre).cuda(), torch.from_numpy(ext).cuda()

    def call():
        sgl.sgl_extend_attn(q, kd, vd, table, pre_d, ext_d, p, o, lse, ws)

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    sgl.sgl_check(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    pairs = sum(int(ext[r]) * int(pre[r]) + int(ext[r]) * (int(ext[r]) + 1) // 2 for r in range(len(seqs)))
    flops = 4.0 * w.d * w.Hq * pairs
    tflops = flops / (ms / 1e3) / 1e12

    # the same step with the KV write fused in (new K/V scattered into the
    # pool by the extend kernel itself)
    kf, vf = W.make_new_kv(w, int(ext.sum()))
    kn, vn = W.to_dtype(w, kf).cuda(), W.to_dtype(w, vf).cuda()

    def call_kv():
        sgl.sgl_extend_attn_kvwrite(q, kn, vn, kd, vd, table, pre_d, ext_d, p, o, lse, ws)

    for _ in range(3):
        call_kv()
    torch.cuda.synchronize()
    sgl.sgl_check(ws)
    e0.record()
    for _ in range(steps):
        call_kv()
    e1.record()
    torch.cuda.synchronize()
    ms_kv = e0.elapsed_time(e1) / steps

    # the same step over FP8 (E4M3) copies of the pools (per-tensor scales
    # amax / 448; the new tokens' rows are in the pools as in the bf16 step)
    def q8(x):
        sc = float(x.float().abs().max()) / 448.0
        return W.quantize_e4m3(x, sc), sc
    k8, ks = q8(kd)
    v8, vs = q8(vd)
    p8 = sgl.make_params(sgl.SGL_DTYPE_BF16_FP8KV, len(seqs), w.Hq, w.Hkv, w.d, S, w.page_size, k_scale=ks,
                         v_scale=vs, host_prefix_lens=pre, host_extend_lens=ext)

    def call_fp8():
        sgl.sgl_extend_attn(q, k8, v8, table, pre_d, ext_d, p8, o, lse, ws)

    for _ in range(3):
        call_fp8()
    torch.cuda.synchronize()
    sgl.sgl_check(ws)
    e0.record()
    for _ in range(steps):
        call_fp8()
    e1.record()
    torch.cuda.synchronize()
    ms_f8 = e0.elapsed_time(e1) / steps
    del k8, v8
    return {"workload": EXTEND_WORKLOAD, "tflops": tflops, "ms_per_call": ms, "gflop_per_call": flops / 1e9,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": tflops / bf16_peak, "peak_source": "measured bf16 burst"},
            "tokens_per_s": int(ext.sum()) / (ms / 1e3), "steps": steps,
            "kv_write_fused": {"ms_per_call": ms_kv, "tflops": flops / (ms_kv / 1e3) / 1e12,
                               "kv_bytes_written": int(kn.numel() * 2 * 2)},
            "fp8_kv": {"ms_per_call": ms_f8, "tflops": flops / (ms_f8 / 1e3) / 1e12,
                       "kv_dtype": "e4m3 (per-tensor scales); one K/V stage, codes converted to f16 in shared memory"}}


def bench_fp8(sgl, W, torch, w, kd, vd, inst, steps, hbm_peak, num_sms=0, name=None):
    """The same decode batches on an FP8 (E4M3) copy of the pool: per-tensor
    scales amax / 448, codes from torch's round-to-nearest conversion (input
    preparation only; the decode call reads the codes)."""
    S = kd.shape[0]

    def quant(x):
        amax = float(x.float().abs().max())
        sc = amax / 448.0 if amax > 0 else 1.0
        q = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
        step = 1 << 16
        for i in range(0, x.shape[0], step):
            q[i:i + step] = W.quantize_e4m3(x[i:i + step], sc)
        return q, sc

    k8, ks = quant(kd)
    v8, vs = quant(vd)
    per_tok = 2 * w.Hkv * w.d
    calls = []
    for it in inst:
        gnp = sgl.groups_as_numpy(sgl.sgl_groups_view(it["groups"]))
        p = sgl.make_params(sgl.SGL_DTYPE_BF16_FP8KV, it["B"], w.Hq, w.Hkv, w.d, S, w.page_size, num_sms=num_sms,
                            k_scale=ks, v_scale=vs)
        plan = sgl.sgl_decode_plan(p, it["out"]["seq_lens"], sgl.sgl_groups_view(it["groups"]))
        ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
        sgl.sgl_plan_upload(plan, ws)
        ub = int((gnp["seg_end"] - gnp["seg_begin"]).sum()) * per_tok
        calls.append(dict(it, plan=plan, ws=ws, ub=ub, o=torch.empty_like(it["o"]), lse=torch.empty_like(it["lse"]),
                          streamed=sgl.sgl_plan_info(plan)))
    for s in range(max(3, len(calls))):
        decode_call(sgl, k8, v8, calls[s % len(calls)])
    torch.cuda.synchronize()
    for c in calls:
        sgl.sgl_check(c["ws"])
    n = max(len(calls), steps - steps % len(calls))
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            for j in range(n):
                decode_call(sgl, k8, v8, calls[j % len(calls)])
    torch.cuda.current_stream().wait_stream(st)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    for c in calls:
        sgl.sgl_check(c["ws"])
    ms = e0.elapsed_time(e1) / n
    ub = sum(c["ub"] for c in calls) / len(calls)
    gbs = ub / (ms / 1e3) / 1e9
    del k8, v8
    torch.cuda.empty_cache()
    return {"workload": name or DECODE_WORKLOAD, "kv_dtype": "e4m3 (per-tensor scales)", "ms_per_call": ms,
            "unique_kv_bytes_per_call": int(ub), "unique_kv_gbs": gbs, "frac_of_hbm": gbs / hbm_peak,
            "tokens_per_s": inst[0]["B"] / (ms / 1e3), "calls_timed": n,
            "path": "same plan as bf16: prefixes shared by many requests on tcgen05 tiles (codes converted to f16 in shared memory), the rest streamed (codes straight into MMA fragments)"}


def bench_mla(sgl, W, torch, steps, bf16_peak, hbm_peak, num_sms=0):
    """MLA grouped decode on the mla_decode batch (Hq 16 over one 576-element
    stored row per token, the Llama-3-8B batch structure), rotating over 4
    batch instances; CUDA-graph loop, CUDA events."""
    w = W.get("mla_decode")
    order, KV = W.make_mla_pool(w)
    S = KV.shape[0]
    kvd = KV.cuda()
    del KV
    tree = sgl.sgl_tree_create(S, w.page_size, order)
    calls = []
    for i in range(4):
        b = W.make_batch(w, i)
        seqs = b.all_tokens()
        groups = sgl.sgl_groups_create()
        out = sgl.sgl_build_batch(tree, seqs, groups=groups)
        gnp = sgl.groups_as_numpy(sgl.sgl_groups_view(groups))
        p = sgl.make_mla_params(len(seqs), w.Hq, S, page_size=w.page_size, num_sms=num_sms)
        plan = sgl.sgl_mla_decode_plan(p, out["seq_lens"], sgl.sgl_groups_view(groups))
        ws = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
        sgl.sgl_plan_upload(plan, ws)
        q = W.to_dtype(w, b.q).cuda()
        calls.append(dict(q=q, table=torch.from_numpy(out["req_to_token"]).cuda(),
                          seq=torch.from_numpy(out["seq_lens"]).cuda(), plan=plan, ws=ws, groups=groups,
                          o=torch.empty(len(seqs), w.Hq, w.dv, dtype=torch.bfloat16, device="cuda"),
                          lse=torch.empty(len(seqs), w.Hq, dtype=torch.float32, device="cuda"),
                          ub=int((gnp["seg_end"] - gnp["seg_begin"]).sum()) * w.d * 2,
                          flops=2.0 * int(out["seq_lens"].sum()) * w.Hq * (w.d + w.dv), B=len(seqs)))
        for r in range(len(seqs)):
            sgl.sgl_tree_finish(tree, int(out["last_nodes"][r]), out["req_to_token"][r], len(seqs[r]))

    def call(c):
        sgl.sgl_mla_decode_attn(c["q"], kvd, c["table"], c["seq"], c["plan"], c["o"], c["lse"], c["ws"])

    for c in calls:
        call(c)
    torch.cuda.synchronize()
    for c in calls:
        sgl.sgl_check(c["ws"])
    n = max(len(calls), steps - steps % len(calls))
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            for j in range(n):
                call(calls[j % len(calls)])
    torch.cuda.current_stream().wait_stream(st)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    for c in calls:
        sgl.sgl_check(c["ws"])
    ms = e0.elapsed_time(e1) / n
    ub = sum(c["ub"] for c in calls) / len(calls)
    fl = sum(c["flops"] for c in calls) / len(calls)
    info = sgl.sgl_plan_info(calls[0]["plan"])
    tf = fl / (ms / 1e3) / 1e12
    return {"workload": "mla_decode", "heads": "Hq16 / one 576-element row (512 latent + 64 position), bf16",
            "batch": calls[0]["B"], "ms_per_call": ms, "unique_kv_bytes_per_call": int(ub),
            "unique_kv_gbs": ub / (ms / 1e3) / 1e9, "frac_of_hbm": ub / (ms / 1e3) / 1e9 / hbm_peak,
            "attention_tflops": tf,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": tf / bf16_peak, "peak_source": "measured bf16 burst (tcgen05 / cuBLAS)"},
            "items": info["num_items"], "chunk_tokens": info["chunk_tokens"], "calls_timed": n,
            "tokens_per_s": calls[0]["B"] / (ms / 1e3)}


def bench_scheduling(sgl, W, w):
    """Cache-aware scheduling simulation (host, native tree) on two traces
    shaped like the lecture notes' demos: few-shot serving (8 applications
    with 2000-token system prompts, 600 requests arriving together) and
    multi-turn chat (300 conversations x 6 turns on a 500-token system
    prompt, 5-20 rounds between turns, a pool too small for every history).
    Per policy: cache hit rate, prefill tokens computed, their KV bytes
    (Llama-3-8B shape, one layer) and the simulation's host time."""
    import numpy as np
    per_tok = kv_bytes_per_token(w)
    traces = {
        "few_shot": (W.few_shot_trace(apps=8, sys_len=2000, n_requests=600, question=(50, 200), output=(50, 200)),
                     1 << 20),
        "multi_turn": (W.multi_turn_trace(conversations=300, turns=6, sys_len=500, user=(50, 150),
                                          output=(50, 200), delay=(5, 20)), 1 << 18),
    }
    policies = {"fcfs_insert_at_prefill": (sgl.SGL_SCHED_FCFS, sgl.SGL_INSERT_AT_PREFILL, 0),
                "lpm_insert_at_prefill": (sgl.SGL_SCHED_LPM, sgl.SGL_INSERT_AT_PREFILL, 64),
                "lpm_insert_at_finish": (sgl.SGL_SCHED_LPM, sgl.SGL_INSERT_AT_FINISH, 64)}
    out = {}
    for name, (reqs, S) in traces.items():
        res = {}
        for pname, (pol, ins, defer) in policies.items():
            order = np.random.default_rng([S, 11]).permutation(S).astype(np.int32)
            tree = sgl.sgl_tree_create(S, 1, order)
            t0 = time.perf_counter()
            _, st = sgl.sgl_sim_run(tree, reqs, policy=pol, insert_at=ins, prefill_budget=2048, max_running=256,
                                    defer_tokens=defer)
            el = time.perf_counter() - t0
            sgl.sgl_tree_destroy(tree)
            res[pname] = {"hit_rate": st["cached_tokens"] / max(1, st["prompt_tokens"]),
                          "prefill_tokens": st["prefill_tokens"], "prefill_kv_bytes": st["prefill_tokens"] * per_tok,
                          "evicted_tokens": st["evicted_tokens"], "rounds": st["rounds"],
                          "host_ms": el * 1e3, "host_us_per_round": el * 1e6 / max(1, st["rounds"])}
        out[name] = {"requests": len(reqs), "pool_slots": S, "prefill_budget": 2048, "max_running": 256,
                     "policies": res}
    return out


def profile_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if one matches the current kernel."""
    path = os.path.join(ROOT, "profiles", "decode_llama3_8b_traffic.json")
    try:
        d = json.load(open(path))
        if d.get("kernel_source_hash") == _kernel_hash():
            return d.get("dram_bytes_per_call")
    except Exception:
        pass
    return None


def _kernel_hash():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "radixattention_prefix_shared_radix_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
