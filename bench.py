#!/usr/bin/env python3
"""Benchmark of the ForwardPass hot path on one GB300 (or N independent
replicas, one per GPU, under torchrun).

Workload (the decode batch): 64 lanes x 1 row, 32 q / 8 kv heads, head_dim
128, bf16, 16-slot pages randomly permuted in a 65,536-page pool, cached
length C ~ U[512, 4096] per lane.  One step is one full pass of the hot path
for the next token of every lane: plan (host metadata -> device work lists),
RoPE + slot scatter, split-KV attention + combine + readout, fold (all).
Step t puts each lane's row at position/slot C+t and reads C+t+1 slots.

Reported (one JSON line on rank 0):
  value        attended tokens/s (sum over rows of visible slots), inputs
               resident in HBM, CUDA events around exactly K steps;
  e2e          the same metric with q/k/v copied from pinned host memory and
               the readout copied back to the host inside every step;
  roofline     achieved HBM GB/s of the split-KV attention kernel
               (algorithmic bytes / its duration, from CUDA events that the
               library records on the launch stream right around it) against
               the measured copy bandwidth; the whole attend call (kernel +
               combine) is reported beside it;
  cpu_baseline the CPU oracle on a bounded sample of the same workload.
`--impl reference` times the CPU oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "attended tokens/s; decode HBM GB/s and prefill TFLOP/s as % of GB300 roofline"
UNIT = "attended tokens/s"
WORKLOAD = "decode_batch"
PROFILE = os.path.join(ROOT, "profiles", "attend_decode_batch.md")
KERNEL_SRC = os.path.join(ROOT, "programmable_paged_kv_gb300", "csrc", "attend_decode_mma.cu")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--workload", default="decode_batch",
                    choices=["decode_batch", "guidance_prefill", "spec_verify", "masked_window",
                             "masked_tova", "masked_decode_window", "masked_decode_tova",
                             "decode_pass", "readout_topk", "decode_loop",
                             "adapters_decode", "adapters_prefill", "batcher"],
                    help="decode_batch (default) is the benchmark line; the others time one "
                         "pass of another configuration")
    ap.add_argument("--no-side-workloads", action="store_true",
                    help="leave out the other configurations' figures from the default line")
    ap.add_argument("--pool-pages", type=int, default=65536,
                    help="pages per K/V pool (smaller pools serve profiler captures)")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl"
        try:
            import torch
            if not torch.cuda.is_available():
                backend = "gloo"
        except Exception:
            backend = "gloo"
        dist.init_process_group(backend)
        pg = dist
    return ws, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ accounting
def attended_tokens(p) -> int:
    """Sum over rows of |visible slots| for a default-visibility pass."""
    lane = np.repeat(np.arange(p.num_lanes), np.diff(p.row_indptr))
    kv = p.kv_len[lane].astype(np.int64)
    return int(np.minimum(kv, p.slots.astype(np.int64) + 1).sum())


def attend_alg_bytes(p, desc) -> int:
    """Algorithmic bytes of one attention call: each distinct visible KV slot
    read once per kv head (K and V), q_rot read, readout rows written (+lse),
    page-table entries of the touched pages."""
    b = W.ELEM_BYTES[desc.dtype]
    d, hq, hkv = desc.head_dim, desc.num_q_heads, desc.num_kv_heads
    kv_slots = int(p.kv_len.astype(np.int64).sum())
    pages = int(sum((int(k) + desc.page_size - 1) // desc.page_size for k in p.kv_len))
    R = p.num_lanes
    return (kv_slots * hkv * 2 * d * b + p.num_rows * hq * d * b + R * hq * (d * b + 4)
            + pages * 4)


def step_alg_bytes(p, desc) -> int:
    b = W.ELEM_BYTES[desc.dtype]
    d, hq, hkv = desc.head_dim, desc.num_q_heads, desc.num_kv_heads
    n = p.num_rows
    append = n * (hq + 2 * hkv) * d * b + n * hq * d * b + n * 2 * hkv * d * b
    return append + attend_alg_bytes(p, desc)


# ------------------------------------------------------------------ peaks / clocks / traffic
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        j = json.load(open(path))
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def peaks_tensor() -> float:
    """Measured dense bf16 TFLOP/s (burst: the kernels are timed alone)."""
    try:
        return float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"])
    except Exception:
        return 1900.0


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"pie_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def profiled_traffic():
    """DRAM bytes per attention launch from the committed ncu summary, if it
    was taken on the current kernel source (else None)."""
    try:
        txt = open(PROFILE).read()
    except OSError:
        return None
    src_hash = hashlib.sha256(open(KERNEL_SRC, "rb").read()).hexdigest()[:16]
    m = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", txt)
    t = re.search(r"dram_bytes_per_attend_call:\s*([0-9]+)", txt)
    if not m or not t or m.group(1) != src_hash:
        return None
    return int(t.group(1))


# ------------------------------------------------------------------ CPU oracle
_ORACLE_SC = {}


def _oracle_scenario(seed: int):
    """The decode batch the oracle is timed on (built once per seed)."""
    if seed not in _ORACLE_SC:
        _ORACLE_SC[seed] = W.decode_batch(seed, lanes=64)
    return _ORACLE_SC[seed]


def oracle_rate(seed: int, seconds: float, threads: int = 0):
    """The oracle on whole decode-batch passes for about `seconds`: attended
    tokens/s with its (lane, kv head) pairs over `threads` host threads (0:
    every core)."""
    import oracle as O
    sc = _oracle_scenario(seed)
    p = sc.passes[0]
    cores = threads or os.cpu_count() or 1
    cp = sc.compact_page_ids(p.page_ids)
    tok = attended_tokens(p)
    total, passes = 0.0, 0
    while total < seconds or passes == 0:
        k, v, fr = sc.k_init.copy(), sc.v_init.copy(), sc.frozen_len0.copy()
        ts = time.perf_counter()
        r = O.run_pass(sc.desc, p, k, v, fr, page_ids=cp, num_threads=cores)
        total += time.perf_counter() - ts
        assert r["err"] == O.OK
        passes += 1
    return tok * passes / total, cores, passes, total


def headline_config(pool_pages: int) -> dict:
    """The decode-batch configuration both arms report."""
    return {"workload": WORKLOAD, "lanes": 64, "rows_per_lane": 1, "q_heads": 32,
            "kv_heads": 8, "head_dim": 128, "page_size": 16, "pool_pages": pool_pages,
            "kv_len": "C+t+1 at step t, C~U[512,4096]",
            "l2": "inputs larger than L2 (~600 MB of KV read per step)",
            "step": "plan+append_kv+attend+fold"}


def run_reference(args, ws, rank):
    """The oracle as the reference arm: step t is decode step t of the
    decode batch (each lane's row at slot C+t, C+t+1 slots read, folded),
    the steps applied in order to one pool, on every host core."""
    if rank != 0:
        return
    import oracle as O
    O.build()
    sc = W.decode_loop(args.seed, lanes=64, steps=args.warmup + args.steps)
    k, v, fr = sc.k_init.copy(), sc.v_init.copy(), sc.frozen_len0.copy()
    cores = os.cpu_count() or 1
    cp = sc.compact_page_ids(sc.passes[0].page_ids)
    times, tok = [], 0
    for t, p in enumerate(sc.passes):
        ts = time.perf_counter()
        r = O.run_pass(sc.desc, p, k, v, fr, page_ids=cp, num_threads=cores)
        dt = time.perf_counter() - ts
        assert r["err"] == O.OK
        if t >= args.warmup:
            times.append(dt)
            tok += attended_tokens(p)
    el = sum(times)
    val = tok / el
    sample = ("decode steps of the decode batch (64 lanes x 1 row, step t at slot C+t), one "
              "full pass per step, all host cores")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": headline_config(args.pool_pages),
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


# ------------------------------------------------------------------ GPU arm
def run_ours(args, ws, rank, local, pg):
    import torch
    from programmable_paged_kv_gb300 import (ForwardPlan, build, make_desc, make_meta, runner,
                                             set_timing_events)
    from programmable_paged_kv_gb300.abi import load
    torch.cuda.set_device(local)
    build()
    load()
    K, Wm = args.steps, args.warmup
    total_steps = 4 * K + 2 * Wm + 2  # warm-up, timed, instrumented (twice), end-to-end
    NP = args.pool_pages
    desc, C, lane_pages, pass_meta = W.decode_loop_meta(seed=args.seed + rank, steps=total_steps,
                                                        num_pool_pages=NP)
    cdesc = make_desc(desc)
    dev = torch.device("cuda", local)
    torch.manual_seed(1000 + args.seed + rank)
    shape = (NP, desc.num_kv_heads, desc.page_size, desc.head_dim)
    k_pool = torch.randn(shape, dtype=torch.bfloat16, device=dev)
    v_pool = torch.randn(shape, dtype=torch.bfloat16, device=dev)
    frozen = torch.from_numpy(C.copy()).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    L, Hq, Hkv, D = 64, desc.num_q_heads, desc.num_kv_heads, desc.head_dim
    NB = 4  # distinct q/k/v batches cycled through the steps
    q_d = [torch.randn((L, Hq, D), dtype=torch.bfloat16, device=dev) for _ in range(NB)]
    k_d = [torch.randn((L, Hkv, D), dtype=torch.bfloat16, device=dev) for _ in range(NB)]
    v_d = [torch.randn((L, Hkv, D), dtype=torch.bfloat16, device=dev) for _ in range(NB)]
    q_rot = torch.empty((L, Hq, D), dtype=torch.bfloat16, device=dev)
    out = torch.empty((L, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((L, Hq), dtype=torch.float32, device=dev)
    # metadata and accounting of every step, prepared before any timed region
    passes = [pass_meta(t) for t in range(total_steps)]
    metas = [make_meta(p, NP) for p in passes]
    acct = [(attended_tokens(p), step_alg_bytes(p, desc), attend_alg_bytes(p, desc))
            for p in passes]
    from programmable_paged_kv_gb300 import workspace_bytes
    ws_bytes = max(workspace_bytes(cdesc, m) for m in metas)  # not monotone in the step
    # two plan workspaces: step t's metadata upload (on a copy stream) overlaps
    # step t-1's kernels; a workspace is rewritten only after the step that
    # used it two steps earlier has finished on the compute stream
    workspaces = [torch.empty(ws_bytes + 4096, dtype=torch.uint8, device=dev) for _ in range(2)]
    stream = torch.cuda.current_stream(dev)
    copy_stream = torch.cuda.Stream(dev)
    ws_free = [torch.cuda.Event(), torch.cuda.Event()]
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    # the attention kernel alone (recorded by the library around its launch)
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    live = []

    def step(t, q, k, v, timed_ev=None, kernel_ev=None, o=None, lo=None):
        i = t % 2
        o = out if o is None else o
        lo = lse if lo is None else lo
        copy_stream.wait_event(ws_free[i])
        plan = ForwardPlan(cdesc, metas[t], workspace=workspaces[i], stream=copy_stream)
        uploaded = torch.cuda.Event()
        uploaded.record(copy_stream)
        stream.wait_event(uploaded)
        # the stream is passed explicitly: looking up torch's current stream
        # costs a few microseconds of host time per call
        plan.append_kv(q, k, v, q_rot, k_pool, v_pool, frozen, status, stream=stream)
        if timed_ev is not None:
            timed_ev[0].record(stream)
        if kernel_ev is not None:
            set_timing_events(*kernel_ev)
        plan.attend(q_rot, k_pool, v_pool, None, o, lo, None, None, status, stream=stream)
        if kernel_ev is not None:
            set_timing_events()
        if timed_ev is not None:
            timed_ev[1].record(stream)
        plan.fold(frozen, None, status, stream=stream)
        ws_free[i].record(stream)
        live.append(plan)
        if len(live) > 4:
            live.pop(0).close()

    t = 0
    for _ in range(Wm):
        step(t, q_d[t % NB], k_d[t % NB], v_d[t % NB])
        t += 1
    torch.cuda.synchronize()
    barrier(pg)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    tokens = 0
    bytes_step = 0
    bytes_attend = 0
    t_start.record(stream)
    for i in range(K):
        tokens += acct[t][0]
        bytes_step += acct[t][1]
        step(t, q_d[t % NB], k_d[t % NB], v_d[t % NB])
        t += 1
    t_end.record(stream)
    torch.cuda.synchronize()
    # 2K more steps, instrumented: K with events around the attend call (its
    # kernels still launching behind one another as they do untimed), then K
    # with the library's events around the attention kernel alone.  Events
    # between kernels stop each from starting while the one before drains, so
    # the step throughput above is taken without them.  A sleep kernel first
    # lets the host queue the steps, so the events time the GPU's work, not
    # host gaps.
    torch.cuda._sleep(int(2 * K * 1e6))
    bytes_call = 0
    for i in range(K):
        bytes_call += acct[t][2]
        step(t, q_d[t % NB], k_d[t % NB], v_d[t % NB], ev[i], None)
        t += 1
    for i in range(K):
        bytes_attend += acct[t][2]
        step(t, q_d[t % NB], k_d[t % NB], v_d[t % NB], None, kev[i])
        t += 1
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(pg)
    el_ms = t_start.elapsed_time(t_end)
    attend_ms = [a.elapsed_time(b) for a, b in ev]
    kernel_ms = [a.elapsed_time(b) for a, b in kev]
    el_max = max_over_ranks(pg, el_ms)
    tokens_all = sum_over_ranks(pg, tokens)
    value = tokens_all / (el_max / 1e3)
    st = int(status.item())

    # ---- end to end: host q/k/v in, readout back to host, every step
    # each step's q, k and v packed in one pinned host buffer (one copy in), the
    # whole pass through one pie_fwd_forward call (plan, append, attend, fold),
    # its readout and lse from one device buffer (one copy out); all on one
    # stream, so a step's copy in follows the previous step's kernels and the
    # host runs ahead of the GPU
    from programmable_paged_kv_gb300 import forward
    qkv_h = [torch.cat([x.reshape(-1) for x in (q_d[j], k_d[j], v_d[j])]).cpu().pin_memory()
             for j in range(NB)]
    nq, nk = q_d[0].numel(), k_d[0].numel()
    ob, lb = out.numel() * out.element_size(), lse.numel() * lse.element_size()
    qkv_d = torch.empty_like(qkv_h[0], device=dev)
    ins = (qkv_d[:nq].view(q_d[0].shape), qkv_d[nq:nq + nk].view(k_d[0].shape),
           qkv_d[nq + nk:].view(v_d[0].shape))
    res_d = torch.empty(ob + lb, dtype=torch.uint8, device=dev)
    o_e, l_e = res_d[:ob].view(out.dtype).view(out.shape), res_d[ob:].view(lse.dtype).view(lse.shape)
    res_h = [torch.empty(ob + lb, dtype=torch.uint8).pin_memory() for _ in range(2)]
    ws_e = workspaces[0]
    for pl in live:
        pl.close()
    live.clear()
    torch.cuda.synchronize()

    def e2e_step(t):
        qkv_d.copy_(qkv_h[t % NB], non_blocking=True)
        forward(cdesc, metas[t], ws_e, *ins, q_rot, k_pool, v_pool, frozen, None, o_e, l_e,
                None, None, None, status, stream=stream)
        res_h[t % 2].copy_(res_d, non_blocking=True)

    for _ in range(Wm):
        e2e_step(t)
        t += 1
    torch.cuda.synchronize()
    barrier(pg)
    e_tok = 0
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        e_tok += acct[t][0]
        e2e_step(t)
        t += 1
    e1.record(stream)  # after the last result's copy to the host
    torch.cuda.synchronize()
    barrier(pg)
    e_ms = max_over_ranks(pg, e0.elapsed_time(e1))
    e_val = sum_over_ranks(pg, e_tok) / (e_ms / 1e3)
    h2d = qkv_h[0].numel() * qkv_h[0].element_size()
    d2h = res_h[0].numel()
    for pl in live:
        pl.close()

    if rank != 0:
        return
    side = None
    if ws == 1 and not args.no_side_workloads:
        # the headline's 4 GiB pools are not needed any more
        k_pool = v_pool = None
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        side = side_workloads(args.seed, local)
    hbm, peak_kind = peaks()
    att_s = sum(attend_ms) / len(attend_ms) / 1e3
    ker_s = sum(kernel_ms) / len(kernel_ms) / 1e3
    achieved = (bytes_attend / K) / ker_s / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": Wm,
        "ms_per_step": el_max / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": headline_config(NP),
        "gpu_launches": 4 * K,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": profiled_traffic(),
                     "kernel": "attend_decode_mma_kernel (split-KV attention on warp-level "
                               "tensor-core MMAs; events recorded "
                               "by the library around its launch)",
                     "peak_kind": peak_kind, "alg_bytes_per_launch": bytes_attend / K,
                     "launch_ms": ker_s * 1e3,
                     "attend_call_ms": att_s * 1e3,
                     "attend_call_frac": (bytes_call / K) / att_s / 1e9 / hbm,
                     "step_alg_gbs": (bytes_step / K) / (el_max / K / 1e3) / 1e9},
        "e2e": {"value": e_val, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "status": st,
    }
    if clk:
        line["clocks"] = clk
    if side:
        g = side["guidance_prefill"]
        tf = peaks_tensor()
        line["roofline_prefill"] = {
            "bound": "tensor", "achieved": g["kernel_tflops"], "peak": tf, "unit": "TFLOP/s",
            "frac": g["kernel_tflops"] / tf, "traffic": None,
            "kernel": "attend_tc_kernel (tcgen05 attention, guidance-pair prefill: 64 lanes x "
                      "64 rows over a shared 1,024-slot prefix; events recorded by the library "
                      "around its launch)",
            "peak_kind": "measured bf16 burst" if tf != 1900.0 else "fallback",
            "alg_flops_per_launch": g["alg_flops"], "launch_us": g["kernel_us"]}
        line["workloads"] = side
    if ws == 1 and not args.no_cpu_baseline:
        import oracle as O
        O.build()
        rate, cores, passes, secs = oracle_rate(args.seed, args.cpu_seconds)
        rate1, _, passes1, secs1 = oracle_rate(args.seed, min(args.cpu_seconds, 4.0), threads=1)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"{passes} full decode-batch passes (64 lanes x 1 row, "
                                          f"seed {args.seed}) in {secs:.1f} s on {cores} threads",
                                "single_thread": {"value": rate1, "unit": UNIT, "cores": 1,
                                                  "sample": f"{passes1} passes in {secs1:.1f} s"}}
    print(json.dumps(line))


# ------------------------------------------------------------------ other workloads
def pass_accounting(p, desc):
    """(attended tokens, attention algorithmic bytes, attention FLOPs) of a
    pass with default or mask visibility.  Bytes count each distinct visible
    physical KV slot once per kv head (shared prefix pages once), q_rot read,
    every row's output (o and lse) and the readout rows written, mask words
    and page-table entries read."""
    b = W.ELEM_BYTES[desc.dtype]
    d, hq, hkv, P = desc.head_dim, desc.num_q_heads, desc.num_kv_heads, desc.page_size
    vis_count = 0
    phys = []
    mask_bytes = 0
    for l in range(p.num_lanes):
        r0, r1 = int(p.row_indptr[l]), int(p.row_indptr[l + 1])
        kv = int(p.kv_len[l])
        if r1 == r0 or kv == 0:
            continue
        if p.mask_word_indptr is None:
            ext = np.minimum(kv, p.slots[r0:r1].astype(np.int64) + 1)
            vis_count += int(ext.sum())
            lane_vis = np.arange(int(ext.max()))
        else:
            nw = (kv + 31) // 32
            union = np.zeros(nw, np.uint32)
            for r in range(r0, r1):
                w = p.mask_words[p.mask_word_indptr[r]:p.mask_word_indptr[r] + nw].copy()
                if kv % 32:
                    w[-1] &= np.uint32((1 << (kv % 32)) - 1)
                vis_count += int(np.unpackbits(w.view(np.uint8)).sum())
                union |= w
            mask_bytes += (r1 - r0) * nw * 4
            bits = np.unpackbits(union.view(np.uint8), bitorder="little")[:kv]
            lane_vis = np.nonzero(bits)[0]
        pages = p.page_ids[p.page_indptr[l]:p.page_indptr[l + 1]].astype(np.int64)
        phys.append(pages[lane_vis // P] * P + lane_vis % P)
    distinct = int(np.unique(np.concatenate(phys)).size) if phys else 0
    R = p.readout.size if p.readout is not None else int((np.diff(p.row_indptr) > 0).sum())
    npages = int(sum((int(k) + P - 1) // P for k in p.kv_len))
    byts = (distinct * hkv * 2 * d * b + p.num_rows * hq * d * b + R * hq * (d * b + 4)
            + p.num_rows * hq * (d * b + 4) + mask_bytes + npages * 4)
    flops = 4 * d * hq * vis_count
    return vis_count, byts, flops


WORKLOADS = {
    "guidance_prefill": lambda s: W.guidance_pairs(s, decodes=0),
    "spec_verify": lambda s: W.spec_verify(s),
    "masked_window": lambda s: W.masked_long(s, "window"),
    "masked_tova": lambda s: W.masked_long(s, "tova"),
    "masked_decode_window": lambda s: W.masked_long(s, "window", rows=1),
    "masked_decode_tova": lambda s: W.masked_long(s, "tova", rows=1),
    "decode_pass": lambda s: W.decode_batch(s),
}


def run_workload(args, local):
    """One JSON line for `--workload W` (see measure_workload)."""
    import torch
    torch.cuda.set_device(local)
    print(json.dumps(measure_workload(args.workload, args.seed, args.steps, args.warmup, local)))


def measure_workload(name, seed, K, Wm, local, device_fill=False):
    """Time one pass of another configuration (first pass of its scenario):
    every row's output and the readout rows; frozen lengths are restored
    before every step so each step is identical.  With device_fill the
    scenario's cached K/V are drawn on the device (same N(0,1) distribution,
    seeded) instead of on the host."""
    import torch
    from programmable_paged_kv_gb300 import (ForwardPlan, build, make_desc, make_meta, runner,
                                             set_timing_events)
    build()
    if device_fill:
        with W.geometry_only():
            sc = WORKLOADS[name](seed)
    else:
        sc = WORKLOADS[name](seed)
    d = sc.desc
    p = sc.passes[0]
    desc = make_desc(d)
    pools = runner.DevicePools(sc, seed=seed)
    frozen0 = torch.from_numpy(sc.frozen_len0.astype(np.int32)).cuda()
    frozen = frozen0.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tdt = torch.bfloat16 if d.dtype == W.BF16 else torch.float32
    N, Hq, D = p.num_rows, d.num_q_heads, d.head_dim
    q = runner.to_device(p.q, d.dtype)
    k = runner.to_device(p.k, d.dtype)
    v = runner.to_device(p.v, d.dtype)
    q_rot = torch.empty((N, Hq, D), dtype=tdt, device="cuda")
    meta = make_meta(p, sc.num_pool_pages)
    from programmable_paged_kv_gb300 import workspace_bytes
    ws = torch.empty(workspace_bytes(desc, meta) + 4096, dtype=torch.uint8, device="cuda")
    plan0 = ForwardPlan(desc, meta, workspace=ws)
    R = plan0.num_readout
    plan0.close()
    out = torch.empty((R, Hq, D), dtype=tdt, device="cuda")
    lse = torch.empty((R, Hq), dtype=torch.float32, device="cuda")
    # every row's attention output (what the next layer of a model reads),
    # besides the readout rows
    out_all = torch.empty((N, Hq, D), dtype=tdt, device="cuda")
    lse_all = torch.empty((N, Hq), dtype=torch.float32, device="cuda")
    mw = None if p.mask_words is None else torch.from_numpy(p.mask_words.view(np.int32)).cuda()
    chan = None if p.channel is None else torch.from_numpy(p.channel.astype(np.int32)).cuda()
    stream = torch.cuda.current_stream()
    live = []
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]

    mev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]

    def step(e=None, ke=None, me=None):
        frozen.copy_(frozen0, non_blocking=True)
        plan = ForwardPlan(desc, meta, workspace=ws)
        if mw is not None:
            # the pass's mask lists, built once for every layer's attend
            if me is not None:
                me[0].record(stream)
            plan.set_mask(mw)
            if me is not None:
                me[1].record(stream)
        plan.append_kv(q, k, v, q_rot, pools.k, pools.v, frozen, status)
        if e is not None:
            e[0].record(stream)
        if ke is not None:
            set_timing_events(*ke)
        plan.attend(q_rot, pools.k, pools.v, mw, out, lse, out_all, lse_all, status)
        if ke is not None:
            set_timing_events()
        if e is not None:
            e[1].record(stream)
        plan.fold(frozen, chan, status)
        live.append(plan)
        if len(live) > 4:
            live.pop(0).close()

    for _ in range(Wm):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(K):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    # 2K more passes, instrumented (events between kernels stop each from
    # starting while the one before drains, so the throughput above is taken
    # without them): K with events around the attend call and the mask step
    # only, so that the call's kernels still launch behind one another as
    # they do untimed, then K with the library's events around the attention
    # kernel alone.  A sleep kernel first lets the host queue the passes, so
    # the events time the GPU's work, not host gaps.  L2 is flushed before
    # each instrumented pass (a 256 MB write, outside its events), so no
    # pass starts with the previous one's K/V cached
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    torch.cuda._sleep(int(2 * K * 1e6))
    for i in range(K):
        flush.fill_(i & 0xFF)
        step(ev[i], None, mev[i])
    for i in range(K):
        flush.fill_(i & 0xFF)
        step(None, kev[i], None)
    torch.cuda.synchronize()
    del flush
    clk = clocks.stop()
    el = t0.elapsed_time(t1) / 1e3
    att = sorted(a.elapsed_time(b) for a, b in ev)
    att_med = att[len(att) // 2] / 1e3
    ker = sorted(a.elapsed_time(b) for a, b in kev)
    ker_med = ker[len(ker) // 2] / 1e3
    msk = sorted(a.elapsed_time(b) for a, b in mev) if mw is not None else [0.0]
    msk_med = msk[len(msk) // 2] / 1e3
    tok, byts, flops = pass_accounting(p, d)
    hbm, kind = peaks()
    tf = peaks_tensor()
    t_roof = max(byts / (hbm * 1e9), flops / (tf * 1e12))
    line = {"workload": name, "metric": METRIC, "unit": UNIT,
            "value": tok * K / el, "ms_per_step": 1e3 * el / K, "steps": K, "warmup": Wm,
            "attend_ms_median": att_med * 1e3, "attended_tokens_per_step": tok,
            "attend_alg_bytes": byts, "attend_alg_flops": flops,
            "attend_hbm_gbs": byts / att_med / 1e9, "attend_hbm_frac": byts / att_med / 1e9 / hbm,
            "attend_tflops": flops / att_med / 1e12, "attend_tensor_frac": flops / att_med / 1e12 / tf,
            "attend_roofline_frac": t_roof / att_med,
            "kernel_ms_median": ker_med * 1e3,
            "mask_lists_ms_median": msk_med * 1e3,
            "kernel_hbm_frac": byts / ker_med / 1e9 / hbm,
            "kernel_tensor_frac": flops / ker_med / 1e12 / tf,
            "status": int(status.item()),
            "peaks": {"hbm_gbs": hbm, "bf16_tflops": tf, "kind": kind}}
    if clk:
        line["clocks"] = clk
    for pl in live:
        pl.close()
    del pools
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return line


# The configurations beside the headline whose figures the default run adds
# to its line: the tensor-core path (prefill TFLOP/s against the bf16 peak)
# and the verify and masked passes.
SIDE_WORKLOADS = ("guidance_prefill", "spec_verify", "masked_window", "masked_tova",
                  "masked_decode_window", "masked_decode_tova")


def side_workloads(seed, local, steps=5, warmup=3):
    """Kernel and call figures of the other configurations, a few passes
    each (inputs drawn on the device), for the default line."""
    out = {}
    for name in SIDE_WORKLOADS:
        r = measure_workload(name, seed, steps, warmup, local, device_fill=True)
        out[name] = {
            "kernel_us": 1e3 * r["kernel_ms_median"], "call_us": 1e3 * r["attend_ms_median"],
            "mask_lists_us_per_pass": 1e3 * r["mask_lists_ms_median"],
            "kernel_tensor_frac": r["kernel_tensor_frac"], "kernel_hbm_frac": r["kernel_hbm_frac"],
            "call_tensor_frac": r["attend_tensor_frac"], "call_hbm_frac": r["attend_hbm_frac"],
            "call_roofline_frac": r["attend_roofline_frac"],
            "kernel_tflops": r["attend_alg_flops"] / (r["kernel_ms_median"] * 1e-3) / 1e12,
            "alg_bytes": r["attend_alg_bytes"], "alg_flops": r["attend_alg_flops"],
            "attended_tokens_per_pass": r["attended_tokens_per_step"],
            "pass_ms": r["ms_per_step"], "steps": steps, "status": r["status"],
            "clocks": r.get("clocks")}
    return out


def run_readout(args, local):
    """Time the readout distribution epilogue: the top-256 tokens of the
    next-token distribution of 64 readout rows over a 128,256-token
    vocabulary (fp32 synthetic logits), p, Z and lse.  Eight distinct logits
    buffers (262 MB, more than L2) are cycled so every step reads from HBM.
    Eager calls give the call time and, through the timing hook, the time of
    the pass over the logits (the stream kernel); the eight calls captured in
    one CUDA graph and replayed give the device time per call without host
    launch costs (`value`)."""
    import torch
    from programmable_paged_kv_gb300 import (build, readout_topk, readout_topk_workspace_bytes,
                                             set_timing_events)
    from programmable_paged_kv_gb300.abi import PIE_F32
    torch.cuda.set_device(local)
    build()
    R, V, K = 64, 128256, 256
    NB = 8
    bufs = [torch.from_numpy(W.readout_logits(args.seed + i, R, V)).cuda() for i in range(NB)]
    ids = torch.empty((R, K), dtype=torch.int32, device="cuda")
    probs = torch.empty((R, K), dtype=torch.float32, device="cuda")
    z = torch.empty(R, dtype=torch.float32, device="cuda")
    lse = torch.empty(R, dtype=torch.float32, device="cuda")
    ws = torch.empty(readout_topk_workspace_bytes(PIE_F32, R, V, K), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    Kst, Wm = args.steps, args.warmup
    for i in range(Wm):
        readout_topk(bufs[i % NB], K, ids, probs, z, lse, workspace=ws)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(Kst)]
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(Kst)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(Kst):
        ev[i][0].record(stream)
        set_timing_events(*kev[i])
        readout_topk(bufs[(Wm + i) % NB], K, ids, probs, z, lse, workspace=ws)
        set_timing_events()
        ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    # device time per call: the NB buffers' calls in one CUDA graph, replayed
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        readout_topk(bufs[0], K, ids, probs, z, lse, workspace=ws)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        for b in bufs:
            readout_topk(b, K, ids, probs, z, lse, workspace=ws)
    g.replay()
    torch.cuda.synchronize()
    reps = max(1, Kst // NB)
    t2 = torch.cuda.Event(enable_timing=True)
    t3 = torch.cuda.Event(enable_timing=True)
    t2.record(stream)
    for _ in range(reps):
        g.replay()
    t3.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    call = sorted(a.elapsed_time(b) for a, b in ev)
    med = call[len(call) // 2] / 1e3
    kms = sorted(a.elapsed_time(b) for a, b in kev)
    kmed = kms[len(kms) // 2] / 1e3
    dev_s = t2.elapsed_time(t3) / 1e3 / (reps * NB)
    byts = R * V * 4 + R * K * 8 + R * 8
    fbytes = R * V * 4          # the stream kernel reads the logits once
    hbm, kind = peaks()
    line = {"workload": "readout_topk", "metric": "readout rows/s (top-256 of a 128,256-token "
            "distribution, p, Z, lse)", "unit": "rows/s", "value": R / dev_s,
            "ms_per_step": dev_s * 1e3, "steps": Kst, "warmup": Wm,
            "device_ms_per_call": dev_s * 1e3, "eager_call_ms_median": med * 1e3,
            "eager_ms_per_step": t0.elapsed_time(t1) / Kst, "eager_rows_per_s": R / med,
            "stream_kernel_ms_median": kmed * 1e3, "alg_bytes": byts,
            "hbm_gbs": byts / dev_s / 1e9, "hbm_frac": byts / dev_s / 1e9 / hbm,
            "gpu_launches": 4 * (Kst + reps * NB),
            "roofline": {"bound": "hbm", "kernel": "stream_kernel",
                         "achieved": fbytes / kmed / 1e9, "peak": hbm, "unit": "GB/s",
                         "frac": fbytes / kmed / 1e9 / hbm, "traffic": None, "peak_kind": kind},
            "config": {"rows": R, "vocab": V, "k": K, "dtype": "f32",
                       "l2": "8 logits buffers cycled (262 MB)"},
            "peaks": {"hbm_gbs": hbm, "kind": kind}}
    if clk:
        line["clocks"] = clk
    print(json.dumps(line))


ADAPTER_SHAPES = {
    # the decode batch's 64 lanes x 1 row, and the guidance-pair prefill's 64
    # lanes x 64 rows, at the q site of a 32 x 128-head model (4096 -> 4096)
    "adapters_decode": dict(rows=[1] * 64, sites=64),
    "adapters_prefill": dict(rows=[64] * 64, sites=8),
}


def adapter_alg_bytes(site) -> int:
    """Bytes one apply must move: x of the adapted rows, y of those rows read
    and written, and A, B, IA3 and scale of every adapter in use (the fp32
    partial sums of A x, about 1% at these sizes, are not counted)."""
    adapted = 0
    for l, a in enumerate(site.adapter_of_lane):
        if a >= 0:
            adapted += int(site.row_indptr[l + 1] - site.row_indptr[l])
    d_in, d_out, r = site.x.shape[1], site.y.shape[1], site.rank
    used = len({int(a) for a in site.adapter_of_lane if a >= 0})
    per_ad = 2 * (r * d_in + d_out * r) + (2 * d_out if site.ia3 is not None else 0) + 4
    return adapted * (2 * d_in + 4 * d_out) + used * per_ad, adapted


def adapter_oracle_rate(site, seconds: float):
    """The oracle on a bounded sample: whole lanes of the same site, repeated
    until `seconds` of CPU time; returns adapted rows per second."""
    import oracle.adapters as OA
    f64 = lambda b: W.bf16_bits_to_f32(b).astype(np.float64)
    x, y, A, B = f64(site.x), f64(site.y), f64(site.lora_a), f64(site.lora_b)
    s = None if site.ia3 is None else f64(site.ia3)
    _, rows = adapter_alg_bytes(site)
    total, reps = 0.0, 0
    while total < seconds or reps == 0:
        t0 = time.perf_counter()
        OA.apply_adapters(x, y, site.row_indptr, site.adapter_of_lane, A, B,
                          site.scale.astype(np.float64), s)
        total += time.perf_counter() - t0
        reps += 1
    return rows * reps / total, reps, total


def blas_threads() -> int:
    """Threads numpy's BLAS may use (all cores when that cannot be read)."""
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def run_adapters(args, local):
    """Time the per-lane adapters at one projection site (LoRA rank 16 and
    IA3, 16 adapters, every 8th lane without one), site after site: `sites`
    distinct sets of weights, x and y (more than L2 together) are cycled, as
    a model's layers would be, so every call reads from HBM."""
    import torch
    from programmable_paged_kv_gb300 import AdapterPlan, build, runner
    torch.cuda.set_device(local)
    build()
    shape = ADAPTER_SHAPES[args.workload]
    sites = [W.adapter_site(args.seed + i, shape["rows"]) for i in range(shape["sites"])]
    dev = lambda a: runner.to_device(a, W.BF16)
    bufs = [(dev(st.x), dev(st.y), dev(st.lora_a), dev(st.lora_b),
             torch.from_numpy(st.scale).cuda(), dev(st.ia3)) for st in sites]
    plan = AdapterPlan(sites[0].row_indptr, sites[0].adapter_of_lane, len(sites[0].scale), 16)
    # every site shares the lanes' adapter ids (one pass, many sites)
    for st in sites[1:]:
        st.adapter_of_lane = sites[0].adapter_of_lane
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    NB, Kst, Wm = len(bufs), args.steps, args.warmup
    for i in range(Wm):
        plan.apply(*bufs[i % NB][:2], *bufs[i % NB][2:], status=status)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(Kst)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(Kst):
        b = bufs[(Wm + i) % NB]
        ev[i][0].record(stream)
        plan.apply(b[0], b[1], b[2], b[3], b[4], b[5], status=status)
        ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    # device time per apply: the NB sites' applies captured in one CUDA graph
    # (host launch costs out of the way) and replayed
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        plan.apply(*bufs[0], status=status)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        for b in bufs:
            plan.apply(*b, status=status)
    g.replay()
    torch.cuda.synchronize()
    reps = max(1, Kst // NB)
    t2 = torch.cuda.Event(enable_timing=True)
    t3 = torch.cuda.Event(enable_timing=True)
    t2.record(stream)
    for _ in range(reps):
        g.replay()
    t3.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert int(status.item()) == 0, f"status {int(status.item())}"
    call = sorted(a.elapsed_time(c) for a, c in ev)
    med = call[len(call) // 2] / 1e3
    dev_s = t2.elapsed_time(t3) / 1e3 / (reps * NB)
    byts, rows = adapter_alg_bytes(sites[0])
    hbm, kind = peaks()
    line = {"workload": args.workload,
            "metric": "adapted rows/s (LoRA r16 + IA3 at a 4096 -> 4096 projection site)",
            "unit": "rows/s", "value": rows / dev_s, "ms_per_step": dev_s * 1e3,
            "steps": Kst, "warmup": Wm, "device_ms_per_apply": dev_s * 1e3,
            "eager_call_ms_median": med * 1e3, "eager_rows_per_s": rows / med,
            "alg_bytes": byts,
            # kernels per apply: one for a grouped plan (a cluster per adapter), else two
            "gpu_launches": (1 if plan.num_groups > 0 else 2) * (Kst + reps * NB),
            "adapter_path": "grouped" if plan.num_groups > 0 else "tiles",
            "roofline": {"bound": "hbm", "achieved": byts / dev_s / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": byts / dev_s / 1e9 / hbm, "traffic": None,
                         "peak_kind": kind},
            "config": {"lanes": len(shape["rows"]), "rows": int(sites[0].row_indptr[-1]),
                       "adapted_rows": rows, "d_in": 4096, "d_out": 4096, "rank": 16,
                       "adapters": 16, "dtype": "bf16", "recipe": sites[0].recipe,
                       "l2": f"{NB} sites cycled "
                             f"({NB * (byts + 2 * 16 * 4096 * 16 * 2) / 1e6:.0f} MB)"}}
    if clk:
        line["clocks"] = clk
    if not args.no_cpu_baseline:
        rate, reps, secs = adapter_oracle_rate(sites[0], min(args.cpu_seconds, 8.0))
        line["cpu_baseline"] = {"value": rate, "unit": "rows/s", "cores": blas_threads(),
                                "kind": "oracle",
                                "sample": f"the whole site, {reps} applies in {secs:.1f} s "
                                          "(numpy fp64 matrix products)"}
    print(json.dumps(line))
    plan.close()


def batcher_closed_loop(trace, steps, max_calls, max_rows, kernel_ms=None):
    """Closed loop of the work-conserving batcher over the ForwardPass: every
    agent (command queue) submits its next decode call only when its previous
    one has completed (an inferlet awaiting its result); on each GPU-idle
    instant one batch is dispatched as one multi-lane pass.  Each agent's
    working set is registered with the batcher once, so a call crosses the
    API boundary as (queue, key, rows, first slot) and a batch's pass is
    built and planned by pie_batcher_plan_forward.  Returns (seconds, calls, batches, attended
    tokens, host seconds by part: dispatch, pass and plan set-up, completion
    and the next submissions)."""
    import torch
    from programmable_paged_kv_gb300 import Batcher, abi, make_desc, runner, set_timing_events
    from programmable_paged_kv_gb300.abi import PieError
    d = trace.pool.desc
    desc = make_desc(d)
    P, Hq, Hkv, D = d.page_size, d.num_q_heads, d.num_kv_heads, d.head_dim
    NP = trace.pool.num_pool_pages
    tdt = torch.bfloat16
    pools = runner.DevicePools(trace.pool)
    b = Batcher([True], max_calls, max_rows)
    Q = len(trace.queue_pages)
    qids = np.asarray([b.add_queue(0) for _ in range(Q)], np.int32)
    for q in range(Q):
        b.set_pages(q, trace.queue_pages[q])  # working set q = agent q
    frozen = np.asarray(trace.cached, np.int32).copy()
    cursor = frozen.astype(np.int64)
    left = np.full(Q, steps, np.int64)
    rng = np.random.default_rng(5)
    # the batch's new rows' q, k, v on the device in pass row order, as a
    # model's projections of the batch would leave them
    q_in = torch.from_numpy(W.f32_to_bf16_bits(rng.standard_normal((Q, Hq, D), dtype=np.float32)).view(np.int16)).cuda().view(tdt)
    kv_in = torch.from_numpy(W.f32_to_bf16_bits(rng.standard_normal((Q, Hkv, D), dtype=np.float32)).view(np.int16)).cuda().view(tdt)
    # pinned staging for each batch's frozen lengths (one asynchronous copy),
    # device buffers for the largest batch, one workspace grown when the
    # planner refuses it
    fr_st = torch.empty(max_calls, dtype=torch.int32).pin_memory()
    fr_np = fr_st.numpy()
    out_h = torch.empty((max_calls, Hq, D), dtype=tdt).pin_memory()
    q_rot_d = torch.empty((max_calls, Hq, D), dtype=tdt, device="cuda")
    out_d = torch.empty((max_calls, Hq, D), dtype=tdt, device="cuda")
    ws = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
    ones = np.ones(Q, np.int64)

    def submit(qs):
        b.submit_forward(qids[qs], qs, ones[:len(qs)], cursor[qs], P)
        cursor[qs] += 1
        left[qs] -= 1

    submit(np.arange(Q))
    ev = [] if kernel_ms is not None else None
    calls = batches = tokens = 0
    host = np.zeros(3)  # dispatch, pass and plan set-up, completion and submission
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    while True:
        h0 = time.perf_counter()
        r = b.dispatch(arrays=True)
        h1 = time.perf_counter()
        host[0] += h1 - h0
        if r is None:
            break
        _, ids, lanes = r
        while True:  # the pass built and planned natively; a refused workspace grows
            try:
                plan, lane_keys, first, kv_len, N = b.plan_forward(ids, lanes, frozen, desc, NP, ws)
                break
            except PieError as e:
                if e.code != abi.PIE_ENOSPACE:
                    raise
                ws = torch.empty(2 * ws.numel(), dtype=torch.uint8, device="cuda")
        L = len(lane_keys)
        fr_np[:L] = frozen[lane_keys]
        fr = fr_st[:L].cuda(non_blocking=True)
        qd, kd = q_in[:N], kv_in[:N]
        host[1] += time.perf_counter() - h1
        q_rot = q_rot_d[:N]
        plan.append_kv(qd, kd, kd, q_rot, pools.k, pools.v, fr)
        out = out_d[:N]
        if ev is not None:
            e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            set_timing_events(*e)
            ev.append(e)
        plan.attend(q_rot, pools.k, pools.v, None, out)
        if ev is not None:
            set_timing_events()
        plan.fold(fr)
        out_h[:N].copy_(out)  # the agents' results (a completion event each)
        plan.close()
        h2 = time.perf_counter()
        frozen[lane_keys] = kv_len  # every new row folded
        tokens += int(kv_len.sum())
        calls += len(ids)
        batches += 1
        b.complete(ids)
        again = lane_keys[left[lane_keys] > 0]  # one call per agent in flight: lane = agent
        if again.size:
            submit(again)
        host[2] += time.perf_counter() - h2
    torch.cuda.synchronize()
    secs = time.perf_counter() - t0
    if ev is not None:
        kernel_ms.extend(a.elapsed_time(c) for a, c in ev)
    b.close()
    return secs, calls, batches, tokens, host


def run_batcher(args, local):
    """The work-conserving batcher in a closed loop (see batcher_closed_loop)
    on the decode batch's shape: 64 agents with C ~ U[512, 4096] cached slots,
    `--steps` decode calls each; batches of up to 64 calls against one call
    per pass."""
    import torch
    import oracle.batcher as OB
    from programmable_paged_kv_gb300 import build
    torch.cuda.set_device(local)
    build()
    steps = min(max(args.steps, 4), 64)  # each agent's pages hold 64 slots past its context
    trace = W.forward_calls(args.seed, queues=64, calls_per_queue=1, prefix=512, private_hi=3584,
                            prefill_lo=64, prefill_hi=64, num_pool_pages=args.pool_pages)
    # warm-up (libraries, allocator, first plans)
    batcher_closed_loop(trace, 2, 64, 4096)
    batcher_closed_loop(trace, 2, 1, 4096)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    kms = []
    secs, calls, batches, tokens, host = batcher_closed_loop(trace, steps, 64, 4096, kms)
    s1, c1, b1, t1, h1 = batcher_closed_loop(trace, steps, 1, 4096)
    clk = clocks.stop()
    # the oracle batcher on the same closed loop's decisions (dispatch + complete)
    ob = OB.Batcher({q: 0 for q in range(64)}, {0: True}, 64, 4096)
    nxt, t_orc, left = 0, 0.0, [steps] * 64
    for q in range(64):
        ob.submit(OB.Call(nxt, q, 0, 1, key=q)); nxt += 1
    while True:
        h0 = time.perf_counter()
        r = ob.dispatch()
        if r is None:
            break
        ob.complete(r.calls)
        t_orc += time.perf_counter() - h0
        for c in r.calls:
            q = ob.calls[c].queue
            left[q] -= 1
            if left[q] > 0:
                ob.submit(OB.Call(nxt, q, 0, 1, key=q)); nxt += 1
    hbm, kind = peaks()
    D, Hkv = 128, 8
    kbytes = tokens * Hkv * 2 * D * 2
    kern = sum(kms) / 1e3
    line = {"workload": "batcher",
            "metric": "forward calls/s, closed loop of 64 decode agents through the "
                      "work-conserving batcher",
            "unit": "calls/s", "value": calls / secs, "ms_per_step": secs / batches * 1e3,
            "steps": steps, "warmup": 2, "higher_is_better": True, "dtype": "bf16",
            "data": "synthetic",
            "one_call_per_pass": {"calls_per_s": c1 / s1, "passes": b1},
            "speedup_vs_one_call_per_pass": (calls / secs) / (c1 / s1),
            "batches": batches, "mean_batch_calls": calls / batches,
            "attended_tokens_per_s": tokens / secs,
            "host_us_per_batch": {"dispatch": host[0] / batches * 1e6,
                                  "pass_and_plan": host[1] / batches * 1e6,
                                  "complete_and_submit": host[2] / batches * 1e6,
                                  "total": host.sum() / batches * 1e6},
            "attention_kernel_ms_per_batch": sum(kms) / len(kms) if kms else None,
            "e2e": {"value": calls / secs, "unit": "calls/s",
                    "h2d_bytes_per_step": 64 * 4,
                    "d2h_bytes_per_step": 64 * 32 * 128 * 2,
                    "inputs": "the batch's q/k/v on the device in pass row order (a model's "
                              "projections of the batch); a batch copies its frozen lengths "
                              "in and the pass's metadata through the planner, and its "
                              "outputs out"},
            "gpu_launches": batches * 5,
            "roofline": {"bound": "hbm", "achieved": kbytes / kern / 1e9 if kern else None,
                         "peak": hbm, "unit": "GB/s",
                         "frac": kbytes / kern / 1e9 / hbm if kern else None, "traffic": None,
                         "kernel": "attention kernels of the batched passes"},
            "config": {"workload": "batcher", "agents": 64, "decode_calls_each": steps,
                       "max_calls": 64, "max_rows": 4096, "q_heads": 32, "kv_heads": 8,
                       "head_dim": 128, "page_size": 16, "cached": "512 shared by pairs + U[0, 3584]",
                       "l2": "KV pages of 64 agents (~300 MB) larger than L2"},
            "cpu_baseline": {"value": batches / t_orc, "unit": "dispatches/s (+complete)",
                             "cores": 1, "kind": "oracle",
                             "sample": f"the oracle batcher on the same closed loop ({batches} "
                                       f"dispatches); the native one took "
                                       f"{host[0] / batches * 1e6:.1f} us per dispatch"}}
    if clk:
        line["clocks"] = clk
    print(json.dumps(line))


def run_decode_loop(args, local):
    """Time the decode loop that runs ahead of the host: the decode batch (64
    lanes, C ~ U[512, 4096]) for K single-token steps in one
    pie_fwd_decode_loop call (geometry and work items from frozen_len on the
    device, no host plan per token), directly and as a replayed CUDA graph of
    the same call (frozen_len reset inside the graph, so every replay is the
    same K steps)."""
    import torch
    from programmable_paged_kv_gb300 import build, decode_loop, decode_loop_workspace_bytes, make_desc
    torch.cuda.set_device(local)
    build()
    K, Wm = args.steps, args.warmup
    NP = args.pool_pages
    d, C, lane_pages, pass_meta = W.decode_loop_meta(seed=args.seed, steps=K + 1, num_pool_pages=NP)
    desc = make_desc(d)
    L, Hq, Hkv, D = 64, d.num_q_heads, d.num_kv_heads, d.head_dim
    p0 = pass_meta(0)
    torch.manual_seed(1000 + args.seed)
    shape = (NP, Hkv, d.page_size, D)
    k_pool = torch.randn(shape, dtype=torch.bfloat16, device="cuda")
    v_pool = torch.randn(shape, dtype=torch.bfloat16, device="cuda")
    q = torch.randn((K, L, Hq, D), dtype=torch.bfloat16, device="cuda")
    k = torch.randn((K, L, Hkv, D), dtype=torch.bfloat16, device="cuda")
    v = torch.randn((K, L, Hkv, D), dtype=torch.bfloat16, device="cuda")
    q_rot = torch.empty((L, Hq, D), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((K, L, Hq, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((K, L, Hq), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    page_indptr = torch.from_numpy(p0.page_indptr.astype(np.int32)).cuda()
    page_ids = torch.from_numpy(p0.page_ids.astype(np.int32)).cuda()
    maxp = int(np.diff(p0.page_indptr).max())
    frozen0 = torch.from_numpy(C.astype(np.int32)).cuda()
    frozen = frozen0.clone()
    ws = torch.empty(decode_loop_workspace_bytes(desc, L, maxp), dtype=torch.uint8, device="cuda")
    tokens = sum(attended_tokens(pass_meta(t)) for t in range(K))
    byts = sum(attend_alg_bytes(pass_meta(t), d) for t in range(K))
    stream = torch.cuda.current_stream()

    def call():
        frozen.copy_(frozen0)
        decode_loop(desc, page_indptr, page_ids, maxp, frozen, q, k, v, q_rot, k_pool, v_pool, out,
                    lse, status, workspace=ws)

    for _ in range(Wm):
        call()
    torch.cuda.synchronize()
    reps = 5
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    direct_s = e0.elapsed_time(e1) / 1e3 / reps
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        call()
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        call()
    g.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    graph_s = e0.elapsed_time(e1) / 1e3 / reps
    hbm, kind = peaks()
    line = {"workload": "decode_loop", "metric": METRIC, "unit": UNIT,
            "value": tokens / graph_s, "value_direct": tokens / direct_s,
            "ms_per_step": graph_s / K * 1e3, "ms_per_step_direct": direct_s / K * 1e3,
            "steps": K, "warmup": Wm, "status": int(status.item()),
            "attend_alg_gbs": byts / graph_s / 1e9, "hbm_frac_whole_step": byts / graph_s / 1e9 / hbm,
            "config": {"lanes": L, "kv_len": "C+t+1, C~U[512,4096]", "pool_pages": NP,
                       "step": "geometry+RoPE/scatter+attend+combine+fold on the device"},
            "peaks": {"hbm_gbs": hbm, "kind": kind}}
    if clk:
        line["clocks"] = clk
    print(json.dumps(line))


def main():
    args = parse()
    ws, rank, local, pg = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    elif args.workload == "readout_topk":
        run_readout(args, local)
    elif args.workload == "decode_loop":
        run_decode_loop(args, local)
    elif args.workload in ADAPTER_SHAPES:
        run_adapters(args, local)
    elif args.workload == "batcher":
        run_batcher(args, local)
    elif args.workload != "decode_batch":
        run_workload(args, local)
    else:
        run_ours(args, ws, rank, local, pg)
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
