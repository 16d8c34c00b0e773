"""Benchmark of the tree-verify step: one tree_attn_verify (one layer) + one tree_accept.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]

Prints one JSON line (rank 0).  Inputs are seeded synthetic stand-ins with the
workload's shapes; they are built once and stay resident in HBM for `value`.
`e2e` repeats the step through the same C-ABI calls with every per-step input
copied in from pinned host memory and the results copied back.  The reference
arm times the float64 CPU oracle on a bounded sample of the same workload.
Multi-GPU runs (torchrun) are independent replicas: weak scaling, no collective
on the data path.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gen  # noqa: E402
from gen import inputs as gi  # noqa: E402

METRIC = "tree-verify steps/s & KV-read HBM GB/s (frac of peak) per batch×prefix×tree"
DEFAULT_WORKLOAD = "c4_llama3_70b_bf16_t0.7"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def algorithmic_work(x: gi.TreeInputs):
    """Bytes and FLOPs one tree_attn_verify must move / do, and the accept bytes."""
    w = x.workload
    eb = 2 if w.dtype == "bf16" else 4
    ntok = x.prefix_lens.astype(np.int64) + w.num_nodes
    kv_bytes = int(ntok.sum()) * w.num_kv_heads * w.head_dim * 2 * eb
    qo_bytes = 2 * w.batch * w.num_nodes * w.num_q_heads * w.head_dim * eb
    pt_bytes = int(((ntok + w.page_size - 1) // w.page_size).sum()) * 4
    attn_bytes = kv_bytes + qo_bytes + pt_bytes
    attn_flops = 4 * w.num_q_heads * w.head_dim * int((w.num_nodes * ntok).sum())
    rows = w.batch * w.num_nodes * w.vocab * 4
    accept_bytes = rows * (1 if w.greedy else 2)
    return dict(kv_bytes=kv_bytes, attn_bytes=attn_bytes, attn_flops=attn_flops, accept_bytes=accept_bytes)


# Every configuration the metric is quoted per (batch x prefix x tree): the five workloads,
# with the Llama-3-70B shape at batches 1, 8 and 32, greedy and at T = 0.7.
SWEEP = ["c1_tiny_f32_greedy", "c2_llama3_8b_bf16_greedy", "c3_llama2_7b_bf16_stoch",
         "c4_llama3_70b_bf16_greedy@b1", "c4_llama3_70b_bf16_t0.7@b1",
         "c4_llama3_70b_bf16_greedy@b8", "c4_llama3_70b_bf16_t0.7@b8",
         "c4_llama3_70b_bf16_greedy", "c4_llama3_70b_bf16_t0.7", "c5_ragged_b64_bf16_stoch"]
KERNEL_NAMES = {1: "attn_simt_kernel", 2: "attn_tc_kernel<false>", 3: "attn_tc_pair_kernel<false>",
                4: "attn_tc_kernel<true>", 5: "attn_tc_pair_kernel<true>"}
L2_FLUSH_BYTES = 512 << 20       # written before every timed call of the sweep: 4x the 129 MB L2


def attn_roofline(work, t_attn_ms, hbm, tf_burst):
    """Achieved rates of one tree_attn_verify and the roof that binds it.  The tensor roof is
    the burst bf16 peak: every timed region here is milliseconds long, at full clock."""
    t = t_attn_ms * 1e-3
    tflops = work["attn_flops"] / t / 1e12
    gbs = work["attn_bytes"] / t / 1e9
    t_tc = work["attn_flops"] / (tf_burst * 1e12)
    t_hbm = work["attn_bytes"] / (hbm * 1e9)
    bound = "tensor" if t_tc > t_hbm else "hbm"
    return dict(bound=bound, tflops=tflops, gbs=gbs, tensor_frac=tflops / tf_burst, hbm_frac=gbs / hbm,
                frac=(tflops / tf_burst) if bound == "tensor" else (gbs / hbm),
                # the largest fraction of HBM the KV reads can reach when the tensor pipe runs at its peak
                kv_frac_cap=min(1.0, work["kv_bytes"] / max(t_tc, t_hbm) / 1e9 / hbm))


def walk_row_bytes(path, alen, parents, vocab, greedy) -> int:
    """Bytes of the rows an accept walk must read: each visited node's target row and, in a
    stochastic walk, the draft row of each visited node at which a child was rejected."""
    rows = 0
    for b_ in range(len(alen)):
        n = int(alen[b_])
        nodes = [0] + [int(c) for c in path[b_, :n]]
        par = parents[b_]
        for i, cur in enumerate(nodes):
            rows += 1
            if greedy:
                continue
            kids = [k for k in range(len(par)) if par[k] == cur]
            if i < n:
                rows += kids[0] != nodes[i + 1]           # the accepted child is not the first
            else:
                rows += len(kids) > 0                     # every child was rejected
    return rows * vocab * 4


def kernel_source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "eagle_speculative_tree_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.startswith("attn_") or f in ("common.cuh", "sm100.cuh", "tree_mask.cu"):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel is unchanged since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        recs = json.load(f)
    for r in recs:
        if r.get("workload") == workload and r.get("kernel") == kernel and \
                r.get("source_digest") == kernel_source_digest():
            return r.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def job_throughput(world: int, steps: int, local_ms: float, device) -> tuple:
    """Whole-job rate of `world` independent replicas that each ran `steps` steps in
    local_ms: the slowest replica's time (max over ranks) bounds the job, and the job did
    world * steps steps.  Returns (max_ms, steps per second)."""
    import torch
    t = local_ms
    if world > 1:
        import torch.distributed as dist
        tt = torch.tensor([local_ms], dtype=torch.float64, device=device)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t = float(tt.item())
    return t, world * steps / (t * 1e-3)


def to_device(x: gi.TreeInputs, dev):
    import torch
    w = x.workload
    bf = w.dtype == "bf16"

    def t(a, bf16=False):
        a = np.ascontiguousarray(a)
        h = torch.from_numpy(a.view(np.int16) if bf16 else a).to(dev)
        return h.view(torch.bfloat16) if bf16 else h

    return dict(q=t(x.q, bf), k=t(x.k_pages, bf), v=t(x.v_pages, bf), pt=t(x.page_table), pl=t(x.prefix_lens),
                par=t(x.tree_parents), lg=t(x.target_logits), tok=t(x.draft_tokens),
                qp=None if w.greedy else t(x.draft_probs), u=None if w.greedy else t(x.uniforms))


def sweep_one(ts, name, dev, stream, steps, warmup, flush, hbm, tf_burst):
    """One configuration: `steps` timed tree_attn_verify + tree_accept pairs, each call timed
    by its own CUDA events with L2 flushed (a 512 MB write) before it."""
    import torch
    w = gen.get(name)
    x = gi.make_inputs(w)
    d = to_device(x, dev)
    out = torch.empty_like(d["q"])
    prob = ts.attn_problem(d["q"], d["k"], d["pt"])
    plan = ts.attn_plan(prob)
    ws_a = torch.empty(ts.attn_workspace_bytes(prob), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(ts.accept_workspace_bytes(w.batch, w.num_nodes, w.vocab), dtype=torch.uint8, device=dev)
    path = torch.empty((w.batch, w.num_nodes), dtype=torch.int32, device=dev)
    alen = torch.empty((w.batch,), dtype=torch.int32, device=dev)
    bonus = torch.empty((w.batch,), dtype=torch.int32, device=dev)

    def attn():
        ts.tree_attn_verify(d["q"], d["k"], d["v"], d["pt"], d["pl"], d["par"], out, workspace=ws_a, stream=stream)

    def acc():
        ts.tree_accept(d["lg"], d["tok"], d["qp"], d["par"], d["u"], w.temperature, accept_path=path,
                       accept_len=alen, bonus_token=bonus, workspace=ws_b, stream=stream)

    for _ in range(warmup):
        attn()
        acc()
    torch.cuda.synchronize()
    if ts.read_status(ws_a) or ts.read_status(ws_b):
        raise RuntimeError(f"{name}: device status flagged an input error")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for e in ev:
        flush.zero_()
        e[0].record(stream)
        attn()
        e[1].record(stream)
        flush.zero_()
        e[2].record(stream)
        acc()
        e[3].record(stream)
    torch.cuda.synchronize()
    ta = np.array([e[0].elapsed_time(e[1]) for e in ev])
    tb = np.array([e[2].elapsed_time(e[3]) for e in ev])
    work = algorithmic_work(x)
    t_attn, t_acc = float(ta.mean()), float(tb.mean())
    roof = attn_roofline(work, t_attn, hbm, tf_burst)
    kv_gbs = work["kv_bytes"] / (t_attn * 1e-3) / 1e9
    lens = alen.cpu().numpy()
    return {"workload": w.name, "batch": w.batch, "tree_nodes": w.num_nodes, "temperature": w.temperature,
            "plan": {"kernel": KERNEL_NAMES[plan.kernel], "num_splits": plan.num_splits, "merge": bool(plan.merge)},
            "t_attn_ms": round(t_attn, 4), "t_attn_p10_p90_ms": [round(float(np.percentile(ta, 10)), 4),
                                                               round(float(np.percentile(ta, 90)), 4)],
            "t_accept_ms": round(t_acc, 4), "steps_per_s": round(1e3 / (t_attn + t_acc), 1),
            "kv_read_gbs": round(kv_gbs, 1), "kv_frac_of_hbm_peak": round(kv_gbs / hbm, 4),
            "attn_tflops": round(roof["tflops"], 1), "tensor_frac": round(roof["tensor_frac"], 4),
            "bound": roof["bound"], "frac": round(roof["frac"], 4), "kv_frac_cap": round(roof["kv_frac_cap"], 4),
            "mean_accept_len": round(float(lens.mean()), 3)}


def run_sweep(ts, dev, stream, steps, warmup):
    import torch
    hbm, tf_burst, _tf_sus, _src = peaks()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    rows = []
    for name in SWEEP:
        rows.append(sweep_one(ts, name, dev, stream, steps, warmup, flush, hbm, tf_burst))
        torch.cuda.empty_cache()
    return {"note": "each call timed alone by CUDA events with L2 flushed before it; steps_per_s = "
                    "1 / (t_attn + t_accept); frac = fraction of the binding roof (burst bf16 tensor peak "
                    "or HBM copy rate, measured)", "steps": steps, "configs": rows}


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    import __graft_entry__
    __graft_entry__.build()
    import eagle_speculative_tree_gb300 as ts

    w = gen.get(args.workload)
    x = gi.make_inputs(w)
    bf = w.dtype == "bf16"

    def t(a, bf16=False, pin=False):
        a = np.ascontiguousarray(a)
        h = torch.from_numpy(a.view(np.int16) if bf16 else a)
        h = h.pin_memory() if pin else h.to(dev)
        return h.view(torch.bfloat16) if bf16 else h

    d = dict(q=t(x.q, bf), k=t(x.k_pages, bf), v=t(x.v_pages, bf), pt=t(x.page_table), pl=t(x.prefix_lens),
             par=t(x.tree_parents), lg=t(x.target_logits), tok=t(x.draft_tokens),
             qp=None if w.greedy else t(x.draft_probs), u=None if w.greedy else t(x.uniforms))
    out = torch.empty_like(d["q"])
    prob = ts.attn_problem(d["q"], d["k"], d["pt"], kernel=args.attn_kernel, num_splits=args.attn_splits)
    plan = ts.attn_plan(prob)
    ws_a = torch.empty(ts.attn_workspace_bytes(prob), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(ts.accept_workspace_bytes(w.batch, w.num_nodes, w.vocab), dtype=torch.uint8, device=dev)
    path = torch.empty((w.batch, w.num_nodes), dtype=torch.int32, device=dev)
    alen = torch.empty((w.batch,), dtype=torch.int32, device=dev)
    bonus = torch.empty((w.batch,), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(inp):
        ts.tree_attn_verify(inp["q"], d["k"], d["v"], inp["pt"], inp["pl"], inp["par"], out,
                            kernel=args.attn_kernel, num_splits=args.attn_splits, workspace=ws_a, stream=stream)
        ts.tree_accept(inp["lg"], inp["tok"], inp["qp"], inp["par"], inp["u"], w.temperature,
                       accept_path=path, accept_len=alen, bonus_token=bonus, mode=args.accept_mode,
                       workspace=ws_b, stream=stream)

    resident = dict(q=d["q"], pt=d["pt"], pl=d["pl"], par=d["par"], lg=d["lg"], tok=d["tok"], qp=d["qp"],
                    u=d["u"])
    for _ in range(args.warmup):
        step(resident)
    torch.cuda.synchronize()
    if ts.read_status(ws_a) or ts.read_status(ws_b):
        raise RuntimeError("device status flagged an input error")

    # ---- device-resident timed region
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    time.sleep(0.3)
    n0 = ts.launch_count()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(K):
        ev[i][0].record(stream)
        ts.tree_attn_verify(resident["q"], d["k"], d["v"], resident["pt"], resident["pl"], resident["par"], out,
                            kernel=args.attn_kernel, num_splits=args.attn_splits, workspace=ws_a, stream=stream)
        ev[i][1].record(stream)
        ts.tree_accept(resident["lg"], resident["tok"], resident["qp"], resident["par"], resident["u"],
                       w.temperature, accept_path=path, accept_len=alen, bonus_token=bonus, mode=args.accept_mode,
                       workspace=ws_b, stream=stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = ts.launch_count() - n0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    attn_ms = [a.elapsed_time(b) for a, b in ev]
    t_attn = float(np.mean(attn_ms))
    total_ms, value = job_throughput(world, K, t_start.elapsed_time(t_end), dev)

    # ---- end to end: per-step inputs from pinned host memory, results back to the host
    # the target rows (and draft rows) stay in pinned host memory: the path-only accept walk
    # reads the rows it visits in place over the CPU-GPU link; everything else is copied in
    host = dict(q=t(x.q, bf, pin=True), pt=t(x.page_table, pin=True), pl=t(x.prefix_lens, pin=True),
                par=t(x.tree_parents, pin=True), tok=t(x.draft_tokens, pin=True),
                u=None if w.greedy else t(x.uniforms, pin=True))
    rows_h = dict(lg=t(x.target_logits, pin=True), qp=None if w.greedy else t(x.draft_probs, pin=True))
    # two sets of device inputs and results: step s+1's inputs are copied in, and step s-1's
    # results copied out, on a second stream while step s computes (every step's copies stay
    # inside the timed region)
    def dev_inputs():
        return dict(q=torch.empty_like(d["q"]), pt=torch.empty_like(d["pt"]), pl=torch.empty_like(d["pl"]),
                    par=torch.empty_like(d["par"]), tok=torch.empty_like(d["tok"]),
                    u=None if w.greedy else torch.empty_like(d["u"]), **rows_h)

    def dev_results():
        return dict(out=torch.empty_like(out), path=torch.empty_like(path), alen=torch.empty_like(alen),
                    bonus=torch.empty_like(bonus))

    def host_results():
        return {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in dev_results().items()}

    dsts, outs, hres = [dev_inputs(), dev_inputs()], [dev_results(), dev_results()], [host_results(), host_results()]
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = sum(v.numel() * v.element_size() for v in hres[0].values())
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    drained = [torch.cuda.Event() for _ in range(2)]
    for ev in computed + drained:
        ev.record(stream)

    def copy_in(i):
        copy_stream.wait_event(computed[i])                 # the last step on buffer i is done with it
        with torch.cuda.stream(copy_stream):
            for k, v in host.items():
                if v is not None:
                    dsts[i][k].copy_(v, non_blocking=True)
        copied[i].record(copy_stream)

    def compute(i):
        stream.wait_event(copied[i])
        stream.wait_event(drained[i])                        # its results buffer has been read out
        inp, res = dsts[i], outs[i]
        ts.tree_attn_verify(inp["q"], d["k"], d["v"], inp["pt"], inp["pl"], inp["par"], res["out"],
                            kernel=args.attn_kernel, num_splits=args.attn_splits, workspace=ws_a, stream=stream)
        ts.tree_accept(inp["lg"], inp["tok"], inp["qp"], inp["par"], inp["u"], w.temperature,
                       accept_path=res["path"], accept_len=res["alen"], bonus_token=res["bonus"],
                       mode=args.accept_mode, workspace=ws_b, stream=stream)
        computed[i].record(stream)

    def copy_out(i):
        copy_stream.wait_event(computed[i])
        with torch.cuda.stream(copy_stream):
            for k, v in outs[i].items():
                hres[i][k].copy_(v, non_blocking=True)
        drained[i].record(copy_stream)

    def e2e_run(n):
        copy_in(0)
        for s_ in range(n):
            i = s_ & 1
            compute(i)
            if s_ + 1 < n:
                copy_in(i ^ 1)
            copy_out(i)
        stream.wait_event(drained[(n - 1) & 1])

    e2e_run(2)
    torch.cuda.synchronize()
    K2 = max(3, min(K, 20))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    e2e_run(K2)
    e1.record(stream)
    torch.cuda.synchronize()
    path.copy_(outs[(K2 - 1) & 1]["path"])
    alen.copy_(outs[(K2 - 1) & 1]["alen"])
    e2e_total_ms, e2e_value = job_throughput(world, K2, e0.elapsed_time(e1), dev)
    # host bytes the walk reads in place: at most the visited target rows and their draft rows
    row_bytes = w.vocab * 4 * (1 if w.greedy else 2)
    in_place = int((alen.to(torch.int64) + 1).sum().item()) * row_bytes

    # ---- the accept walk alone with the rows in pinned host memory, against the link's
    # copy rate: the rows it must fetch are the target row of every visited node and, where
    # a child of that node was rejected, its draft row (each once)
    for _ in range(3):
        ts.tree_accept(rows_h["lg"], d["tok"], rows_h["qp"], d["par"], d["u"], w.temperature, accept_path=path,
                       accept_len=alen, bonus_token=bonus, mode=args.accept_mode, workspace=ws_b, stream=stream)
    torch.cuda.synchronize()
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    for _ in range(K2):
        ts.tree_accept(rows_h["lg"], d["tok"], rows_h["qp"], d["par"], d["u"], w.temperature, accept_path=path,
                       accept_len=alen, bonus_token=bonus, mode=args.accept_mode, workspace=ws_b, stream=stream)
    a1.record(stream)
    torch.cuda.synchronize()
    ip_ms = a0.elapsed_time(a1) / K2
    ip_bytes = walk_row_bytes(path.cpu().numpy(), alen.cpu().numpy(), x.tree_parents, w.vocab, w.greedy)
    n_link = min(256 << 20, rows_h["lg"].numel() * 4)
    src_link = rows_h["lg"].view(-1).view(torch.uint8)[:n_link]
    dst_link = torch.empty(n_link, dtype=torch.uint8, device=dev)
    for _ in range(2):
        dst_link.copy_(src_link, non_blocking=True)
    l0 = torch.cuda.Event(enable_timing=True)
    l1 = torch.cuda.Event(enable_timing=True)
    l0.record(stream)
    for _ in range(5):
        dst_link.copy_(src_link, non_blocking=True)
    l1.record(stream)
    torch.cuda.synchronize()
    link_gbs = 5 * n_link / (l0.elapsed_time(l1) * 1e-3) / 1e9
    del dst_link
    ip_gbs = ip_bytes / (ip_ms * 1e-3) / 1e9
    in_place_accept = {"ms": round(ip_ms, 4), "bytes": ip_bytes, "gbs": round(ip_gbs, 1),
                       "link_copy_gbs": round(link_gbs, 1), "frac_of_link": round(ip_gbs / link_gbs, 3),
                       "note": "tree_accept alone with target and draft rows in pinned host memory; bytes = the "
                               "target row of each visited node + the draft row of each node with a rejected "
                               "child, once each; link_copy_gbs = a 256 MiB pinned host-to-device copy"}

    # ---- KV commit of the accepted paths (not part of the step above): timed on the resident
    # pool with the accepted paths of the last step; it moves rows in place, so it runs last
    new_lens = torch.empty_like(d["pl"])
    ws_c = torch.empty(ts.commit_workspace_bytes(), dtype=torch.uint8, device=dev)
    for _ in range(3):
        ts.tree_kv_commit(d["k"], d["v"], d["pt"], d["pl"], path, alen, new_lens, workspace=ws_c, stream=stream)
    torch.cuda.synchronize()
    c0 = torch.cuda.Event(enable_timing=True)
    c1 = torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for _ in range(K2):
        ts.tree_kv_commit(d["k"], d["v"], d["pt"], d["pl"], path, alen, new_lens, workspace=ws_c, stream=stream)
    c1.record(stream)
    torch.cuda.synchronize()
    commit_ms = c0.elapsed_time(c1) / K2
    if ts.read_status(ws_c):
        raise RuntimeError("KV commit flagged an input error")
    commit_bytes = int(alen.sum().item()) * w.num_kv_heads * w.head_dim * (2 if bf else 4) * 2 * 2

    # ---- draft-tree build for the next step (not part of the step above): the workload's
    # num_steps steps of top-k expansion over the vocabulary, then the rerank to N nodes
    from gen import draft as gdraft
    k_d, steps_d = w.topk, w.num_steps
    M_d = 1 + k_d + (steps_d - 1) * k_d * k_d
    lp0 = torch.from_numpy(gdraft.draft_logprobs(1000 + w.cfg_id, w.batch, 1, w.vocab)).to(dev)
    lpk = torch.from_numpy(gdraft.draft_logprobs(2000 + w.cfg_id, w.batch, k_d, w.vocab)).to(dev)
    npar = torch.zeros((w.batch, M_d), dtype=torch.int32, device=dev)
    ntok = torch.zeros_like(npar)
    nsc = torch.zeros((w.batch, M_d), dtype=torch.float32, device=dev)
    fronts = [torch.empty((w.batch, k_d), dtype=torch.int32, device=dev) for _ in range(2)]
    ws_d = torch.empty(ts.draft_workspace_bytes(w.batch, k_d, k_d), dtype=torch.uint8, device=dev)
    ws_r = torch.empty(256, dtype=torch.uint8, device=dev)
    tp = torch.empty((w.batch, w.num_nodes), dtype=torch.int32, device=dev)
    tt = torch.empty_like(tp)

    def build_tree():
        front = None
        for s_ in range(steps_d):
            out = fronts[s_ & 1]
            ts.tree_draft_step(lp0 if s_ == 0 else lpk, s_, k_d, front, npar, ntok, nsc, out, workspace=ws_d,
                               stream=stream)
            front = out
        ts.tree_rerank(npar, ntok, nsc, w.num_nodes, tp, tt, workspace=ws_r, stream=stream)

    for _ in range(3):
        build_tree()
    torch.cuda.synchronize()
    d0 = torch.cuda.Event(enable_timing=True)
    d1 = torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for _ in range(K2):
        build_tree()
    d1.record(stream)
    torch.cuda.synchronize()
    draft_ms = d0.elapsed_time(d1) / K2
    if ts.read_status(ws_d) or ts.read_status(ws_r):
        raise RuntimeError("draft-tree build flagged an input error")
    draft_bytes = (w.batch * w.vocab * 4) * (1 + (steps_d - 1) * k_d)

    # ---- report
    work = algorithmic_work(x)
    hbm, tf_burst, tf_sus, src = peaks()
    kv_gbs = work["kv_bytes"] / (t_attn * 1e-3) / 1e9
    kernel_name = KERNEL_NAMES[plan.kernel]
    traffic = recorded_traffic(w.name, kernel_name)
    rf = attn_roofline(work, t_attn, hbm, tf_burst)
    if rf["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": round(rf["tflops"], 2), "peak": tf_burst, "unit": "TFLOP/s",
                "frac": round(rf["frac"], 4), "traffic": traffic, "peak_kind": "burst bf16 (of " + src + ")"}
    else:
        roof = {"bound": "hbm", "achieved": round(rf["gbs"], 1), "peak": hbm, "unit": "GB/s",
                "frac": round(rf["frac"], 4), "traffic": traffic, "peak_kind": "HBM copy (of " + src + ")"}
    roof.update({"kernel": f"tree_attn_verify ({kernel_name} + prologue" + (" + merge)" if plan.merge else ")"),
                 "algorithmic_bytes": work["attn_bytes"], "algorithmic_flops": work["attn_flops"],
                 "launch_ms": round(t_attn, 4), "hbm_frac": round(rf["hbm_frac"], 4),
                 "tensor_frac": round(rf["tensor_frac"], 4), "kv_frac_cap": round(rf["kv_frac_cap"], 4),
                 "kv_frac_cap_note": "KV bytes / max(FLOPs / burst tensor peak, bytes / HBM peak) / HBM peak: "
                                     "the KV fraction this workload can reach with the tensor pipe at its peak"})
    ms_step = total_ms / K
    lens = alen.cpu().numpy()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "steps/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (seeded; shapes and distributions of the workload, no model weights)",
        "config": {"workload": w.name, "batch": w.batch, "prefix": [w.prefix_lo, w.prefix_hi],
                   "tree_nodes": w.num_nodes, "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
                   "head_dim": w.head_dim, "page_size": w.page_size, "vocab": w.vocab,
                   "temperature": w.temperature, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2 (KV {work['kv_bytes'] / 1e9:.2f} GB, accept rows "
                         f"{work['accept_bytes'] / 1e9:.2f} GB per step)"},
        "kv_read_gbs": round(kv_gbs, 1), "kv_frac_of_hbm_peak": round(kv_gbs / hbm, 4),
        "kv_frac_cap": round(rf["kv_frac_cap"], 4),
        "t_attn_ms": round(t_attn, 4), "t_accept_ms": round(ms_step - t_attn, 4),
        "attn_plan": {"kernel": kernel_name, "num_splits": plan.num_splits, "split_tokens": plan.split_tokens,
                      "merge": bool(plan.merge)},
        "accept_mode": ["auto", "all rows", "path only"][args.accept_mode],
        "mean_accept_len": round(float(lens.mean()), 3), "tokens_per_step": round(float(lens.mean()) + 1, 3),
        "roofline": roof,
        "e2e": {"value": round(e2e_value, 2), "unit": "steps/s", "h2d_bytes_per_step": h2d,
                "h2d_read_in_place_bytes_per_step_max": in_place,
                "in_place_accept": in_place_accept,
                "note": "q, page table, lengths, parents, tokens, uniforms copied in from pinned host memory and "
                        "attention output + accept results copied back, on a second stream overlapping the "
                        "neighbouring steps' compute; target logits and draft probabilities stay pinned on "
                        "the host and the accept walk reads the visited rows in place",
                "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "kv_commit": {"ms": round(commit_ms, 4), "bytes": commit_bytes,
                      "gbs": round(commit_bytes / (commit_ms * 1e-3) / 1e9, 1),
                      "note": "tree_kv_commit of the step's accepted paths, timed apart from the step"},
        "draft_tree": {"ms": round(draft_ms, 4), "bytes": draft_bytes,
                       "gbs": round(draft_bytes / (draft_ms * 1e-3) / 1e9, 1), "steps": steps_d, "topk": k_d,
                       "note": "tree_draft_step x steps + tree_rerank for the next tree, timed apart from the step"},
        "clocks": clk,
    }
    if world == 1 and not args.no_sweep:
        del d, resident, host, rows_h, dsts, outs, hres
        torch.cuda.empty_cache()
        line["sweep"] = run_sweep(ts, dev, stream, min(K, 20), args.warmup)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


class OracleSample:
    """The float64 oracle on a bounded sample of a workload, scaled to one full step."""

    def __init__(self, w):
        from oracle import accept as oacc
        from oracle import attention as oatt
        self.oacc, self.oatt, self.w = oacc, oatt, w
        self.sample_b = min(2, w.batch)
        self.x = gi.make_inputs(w.with_batch(self.sample_b))
        dt = w.dtype
        self.q, self.kp, self.vp = gi.as_float(self.x.q, dt), gi.as_float(self.x.k_pages, dt), \
            gi.as_float(self.x.v_pages, dt)
        full_prefix = gi.make_inputs(w, with_accept=False, with_attention=False).prefix_lens.astype(np.int64)
        self.full_tok = int((full_prefix + w.num_nodes).sum()) * w.num_kv_heads
        self.pairs = [(b, h) for b in range(self.sample_b) for h in range(w.num_kv_heads)]

    def run(self, budget_s: float):
        w, x = self.w, self.x
        done, t_att = [], 0.0
        for pr in self.pairs:
            t0 = time.perf_counter()
            self.oatt.tree_attention(self.q, self.kp, self.vp, x.page_table, x.prefix_lens, x.tree_parents,
                                     w.page_size, [pr])
            t_att += time.perf_counter() - t0
            done.append(pr)
            if t_att > budget_s * 0.8:
                break
        t0 = time.perf_counter()
        self.oacc.tree_accept(x.target_logits, x.draft_tokens, x.draft_probs, x.tree_parents, x.uniforms,
                              w.temperature)
        t_acc = time.perf_counter() - t0
        samp_tok = sum(int(x.prefix_lens[b]) + w.num_nodes for b, _ in done)
        t_attn_full = t_att * self.full_tok / samp_tok
        t_acc_full = t_acc * w.batch / self.sample_b
        t_step = t_attn_full + t_acc_full
        return {"value": round(1.0 / t_step, 6), "unit": "steps/s", "cores": os.cpu_count(), "kind": "oracle",
                "estimate": "scaled: the sample's measured time x (full step's tokens / sample's tokens); "
                            "the full step itself is not run",
                "sample": f"float64 oracle: attention over {len(done)} (sequence, kv head) pairs and the accept "
                          f"walk over {self.sample_b} sequences, scaled by tokens to the full {w.name} step",
                "t_attn_s_full_step": round(t_attn_full, 3), "t_accept_s_full_step": round(t_acc_full, 3)}


def cpu_baseline(w, budget_s: float = 20.0):
    return OracleSample(w).run(budget_s)


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    w = gen.get(args.workload)
    sampler = OracleSample(w)
    budget = max(0.5, 120.0 / max(1, args.steps + args.warmup))
    per = []
    for i in range(args.warmup + args.steps):
        cb = sampler.run(budget)
        if i >= args.warmup:
            per.append(cb)
    value = float(np.mean([c["value"] for c in per]))
    cb = dict(per[-1])
    cb["value"] = round(value, 6)
    line = {"metric": METRIC, "value": round(value, 6), "unit": "steps/s", "impl": "reference",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1000.0 / value, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "batch": w.batch, "prefix": [w.prefix_lo, w.prefix_hi],
                       "tree_nodes": w.num_nodes, "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
                       "head_dim": w.head_dim, "vocab": w.vocab, "temperature": w.temperature},
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 6), "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(gen.WORKLOADS) +
                    [f"{n}@b{b}" for n in gen.WORKLOADS for b in (1, 2, 8, 16, 32, 64)])
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--attn-kernel", type=int, default=0,
                    help="0 auto, 1 CUDA cores, 2 tensor cores, 3 two query tiles per CTA, 4 CTA pairs")
    ap.add_argument("--attn-splits", type=int, default=0, help="KV splits per (sequence, kv head); 0 = planner")
    ap.add_argument("--accept-mode", type=int, default=0, help="0 auto, 1 all rows, 2 path only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the per-configuration sweep (1 GPU only)")
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
