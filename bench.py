"""Benchmark of one full target-verify step of draft-tree speculative decoding.

A step is one pass of the whole hot path over one synthetic batch:
build_tree_mask -> write_window_kv -> tree_verify_attention (query
rotation, tensor-core pass over prefix and window keys, merge) ->
verify_tree_greedy -> compact_window_rows -> compact_rows. Inputs are resident in HBM when the timed region starts; L2 is
flushed (512 MiB write) before every timed step, outside the step's events.

Default workload: eagle2_p8192_n64 (B=32, Hq=32, Hkv=8, d=128, P=8192, N=64),
the long-prefix regime (P >= 8192) where the attention must reach its
roofline. ``--workload`` picks another.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path shards by request with no exchange); value = all ranks' rows / the
slowest rank's time. ``--impl reference`` times the CPU oracle (fp64 NumPy) on
the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from draft_tree_speculative_gb300 import synth  # noqa: E402

METRIC = "tree-verify attention rows/s & % of HBM/tensor roofline; verify_tree µs/step"
ATTN_SOURCES = ("draft_tree_speculative_gb300/csrc/attention.cu", "draft_tree_speculative_gb300/csrc/tcgen05.cuh",
                "draft_tree_speculative_gb300/csrc/common.cuh")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="eagle2_p8192_n64", choices=list(synth.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-argmax", action="store_true", help="skip the target-argmax measurement")
    ap.add_argument("--no-lanes", action="store_true", help="skip the draft-lane attention measurement")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8-KV attention measurement")
    ap.add_argument("--no-side-workloads", action="store_true",
                    help="skip the long-context and high-concurrency workloads' measurements")
    return ap.parse_args()


# ----------------------------------------------------------------------------
# algorithmic bytes / FLOPs of one tree_verify_attention call
# ----------------------------------------------------------------------------

def attention_work(inp: synth.VerifyInputs):
    w = inp.w
    P = inp.vc.astype(np.int64)
    kv_row = w.Hkv * w.d * 2                      # one slot of K (or V), bf16
    kv = 2 * kv_row * (int(P.sum()) + w.B * w.N)  # prefix + window K and V, read once per KV head
    rows = w.B * w.N * w.Hq
    q = out = rows * w.d * 2
    small = rows * 4 + w.B * w.N * (8 + 4) + inp.layout.page_table.size * 4 + w.B * 4
    bytes_ = kv + q + out + small
    depth_sum = int(inp.depth.sum()) + w.B * w.N
    flops = 4 * w.N * w.Hq * w.d * int(P.sum()) + 4 * w.Hq * w.d * depth_sum
    return bytes_, flops


def attention_roofline(inp, attn_ms, workload):
    """Roofline of one tree_verify_attention call (prep, tree pass, merge) of
    mean CUDA-event duration attn_ms: the slower of the algorithmic bytes at the
    measured HBM bandwidth and the algorithmic FLOPs at the measured sustained
    bf16 rate (the call runs inside a long step)."""
    bytes_, flops = attention_work(inp)
    hbm, tf_burst, tf_sus, src = load_peaks()
    t_hbm = bytes_ / (hbm * 1e9)
    t_mma = flops / (tf_sus * 1e12)
    if t_hbm >= t_mma:
        roof = {"bound": "hbm", "achieved": bytes_ / (attn_ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops / (attn_ms / 1e3) / 1e12, "peak": tf_sus, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = recorded_traffic(workload)
    roof["kernel"] = "tree_verify_attention (attn_prep_kernel + tree_prefix_kernel + tree_merge_kernel)"
    roof["algorithmic_bytes"] = bytes_
    roof["algorithmic_flops"] = flops
    roof["peak_source"] = f"{src} ({'hbm_gbs' if roof['bound'] == 'hbm' else 'bf16_tflops_sustained'})"
    roof["roofline_us"] = max(t_hbm, t_mma) * 1e6
    roof["attention_us"] = attn_ms * 1e3
    return roof


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def attention_source_hash():
    h = hashlib.sha256()
    for rel in ATTN_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per attention call from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("source_hash") != attention_source_hash():
        return None
    return e.get("bytes_per_call")


def load_sm_max_mhz():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f).get("sm_max_mhz", 2070.0))
    return 2070.0


def recorded_instructions(name, workload):
    """Warp instructions per call of a kernel from the committed ncu summary,
    if it was taken on the current source for this workload; else None."""
    p = os.path.join(ROOT, "profiles", "instruction_counts.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        e = json.load(f).get(name)
    src = os.path.join(ROOT, "draft_tree_speculative_gb300", "csrc", "argmax.cu")
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    if not e or e.get("source_hash") != h or e.get("workload") != workload:
        return None
    return e.get("warp_instructions_per_call")


def run_ahead(stream, us=3000.0):
    """Enqueue a GPU spin of about `us` microseconds on `stream`, outside any
    timed events, so that the host enqueues the next steps while it runs and
    the GPU then executes them back to back: device times then measure the
    kernels, not the host's launch latency between small kernels."""
    import torch
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(us * 2000))  # cycles, at about 2 GHz


AHEAD_STEPS = 8  # timed steps enqueued behind each spin


def check_device_error(db, when):
    from draft_tree_speculative_gb300 import device_error_string
    code = int(db.err.item())
    if code:
        raise RuntimeError(f"device reported error {code} during {when}: {device_error_string(code)}")


# ----------------------------------------------------------------------------
# replicas: the slowest rank's time, whole-job throughput
# ----------------------------------------------------------------------------

def reduce_max(x: float, device) -> float:
    """Max of x over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rows_per_s(rows_per_step_per_rank: int, world: int, slowest_ms_per_step: float) -> float:
    """Every rank runs its own replica, so the job's rows per step are world x
    one replica's, and the job is as fast as its slowest rank."""
    return world * rows_per_step_per_rank / (slowest_ms_per_step / 1e3)


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
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
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample
# ----------------------------------------------------------------------------

def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k, "").isdigit():
            return int(os.environ[k])
    return os.cpu_count() or 1


def oracle_sample(inp: synth.VerifyInputs, b: int, nodes):
    """Oracle work for `nodes` of request b: attention rows, the walk and the
    compaction of that request. Returns the number of verify rows done."""
    from oracle import attention as OA
    from oracle import compact as OC
    from oracle import walk as OW
    w = inp.w
    OA.verify_attention(inp.q, inp.k_new, inp.v_new, inp.k_cache, inp.v_cache, inp.layout.page_table, inp.vc,
                        inp.parents, w.Hkv, w.rope_theta, page_size=w.page_size, rows=[(b, v) for v in nodes])
    alen, path, _ = OW.greedy_walk(inp.parents[b], inp.draft[b], inp.target_argmax[b])
    wl = inp.layout.write_locations[b * w.N:(b + 1) * w.N]
    rows = np.arange(w.N)
    kv = [inp.k_cache[wl], inp.v_cache[wl]]
    OC.compact_window_rows(kv, rows, path[None], [alen])
    if inp.hidden is not None:
        OC.compact_hidden_rows(inp.hidden[b * w.N:(b + 1) * w.N], path[None], [alen])
    return len(nodes)


ORACLE_ROWS_PER_SAMPLE = 16  # verify rows (all heads) of one request per oracle sample, in both oracle legs


def cpu_rows_per_s(inp, steps=1, nodes_per_step=ORACLE_ROWS_PER_SAMPLE, min_seconds=0.0, max_steps=100000):
    """The oracle over `steps` samples (or, with min_seconds, as many as fit in
    that time, at most max_steps); each sample is `nodes_per_step` verify rows
    of one request (requests in turn) plus that request's walk and compaction."""
    w = inp.w
    n_nodes = min(nodes_per_step, w.N)
    rows = 0
    done = 0
    t0 = time.perf_counter()
    while done < max_steps and (done < steps or time.perf_counter() - t0 < min_seconds):
        b = done % w.B
        nodes = [(done * n_nodes + k) % w.N for k in range(n_nodes)]
        rows += oracle_sample(inp, b, nodes)
        done += 1
    dt = time.perf_counter() - t0
    return rows / dt, dt, f"{n_nodes} verify rows (all heads) of one request per sample, plus that request's walk " \
                          f"and compaction; {done} sample(s), {rows} rows, {dt:.1f} s"


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank):
    import torch
    from draft_tree_speculative_gb300 import lib
    from draft_tree_speculative_gb300.step import DeviceBatch, run_step

    lib()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = synth.WORKLOADS[args.workload]
    inp = synth.make_inputs(w)
    db = DeviceBatch(inp, device=dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    # prologue (mask + window K/V), attention (prep, tree pass, merge),
    # epilogue (walk + KV and hidden-row compaction): five launches
    names = ("prologue", "attention", "epilogue")
    calls = (db.prologue_step, db.attention_step, db.epilogue_step)
    launches_per_step = DeviceBatch.KERNELS_PER_STEP

    def one_step(ev=None):
        for k, c in enumerate(calls):
            if ev is not None:
                ev[k].record(stream)
            c(stream)
        if ev is not None:
            ev[len(calls)].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1)
            one_step()
    torch.cuda.synchronize()
    check_device_error(db, "warm-up")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        wall0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for s in range(args.steps):
                if s % AHEAD_STEPS == 0:
                    run_ahead(stream)
                flush.fill_(1)
                one_step(events[s])
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    if world > 1:
        torch.distributed.barrier()
    per_call = {n: [] for n in names}
    step_ms = []
    for ev in events:
        step_ms.append(ev[0].elapsed_time(ev[-1]))
        for k, n in enumerate(names):
            per_call[n].append(ev[k].elapsed_time(ev[k + 1]))
    total_ms = reduce_max(sum(step_ms), dev)
    ms_per_step = total_ms / args.steps
    rows_per_step = w.B * w.N
    value = whole_job_rows_per_s(rows_per_step, world, ms_per_step)

    # roofline of the attention call (prep, tree pass, merge)
    attn_ms = statistics.mean(per_call["attention"])
    hbm, tf_burst, tf_sus, src = load_peaks()
    roof = attention_roofline(inp, attn_ms, args.workload)

    # end to end through the public API: pinned host inputs in, result out.
    # A serving loop overlaps the next step's upload with this step's compute:
    # the inputs are double-buffered on the device, each step's upload runs on
    # a copy stream once the step that last used its buffer has finished, and
    # the step waits for its upload. Every step still copies its inputs from
    # pinned host memory and reads its result back inside the timed region.
    e2e = None
    if not args.no_e2e:
        in_names = ("q", "k_new", "v_new", "parents", "depth", "vc", "draft", "target_argmax")
        host = {k: getattr(db, k).cpu().pin_memory() for k in in_names}
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        bufs = [{k: getattr(db, k) for k in in_names}, {k: torch.empty_like(getattr(db, k)) for k in in_names}]
        outs = [(torch.empty_like(db.accept_len, device="cpu").pin_memory(),
                 torch.empty_like(db.accepted_tokens, device="cpu").pin_memory()) for _ in range(2)]
        d2h = outs[0][0].numel() * 4 + outs[0][1].numel() * 4
        copy_stream = torch.cuda.Stream(device=dev)
        ready = [torch.cuda.Event() for _ in range(2)]
        freed = [None, None]

        def pipelined(nsteps):
            for st in range(nsteps):
                i = st % 2
                with torch.cuda.stream(copy_stream):
                    if freed[i] is not None:
                        copy_stream.wait_event(freed[i])
                    for k, t in host.items():
                        bufs[i][k].copy_(t, non_blocking=True)
                    ready[i].record(copy_stream)
                stream.wait_event(ready[i])
                for k in in_names:
                    setattr(db, k, bufs[i][k])
                db.prefix_len = db.vc
                run_step(db, stream)
                with torch.cuda.stream(stream):
                    outs[i][0].copy_(db.accept_len, non_blocking=True)
                    outs[i][1].copy_(db.accepted_tokens, non_blocking=True)
                ev_free = torch.cuda.Event()
                ev_free.record(stream)
                freed[i] = ev_free

        pipelined(args.warmup)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        copy_stream.wait_event(t0)
        pipelined(args.steps)
        t1.record(stream)
        torch.cuda.synchronize()
        for k in in_names:
            setattr(db, k, bufs[0][k])
        db.prefix_len = db.vc
        e_ms = reduce_max(t0.elapsed_time(t1), dev)
        e2e = {"value": whole_job_rows_per_s(rows_per_step, world, e_ms / args.steps), "unit": "rows/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms / args.steps,
               "pipelined": "inputs double-buffered; upload of step k+1 overlaps step k",
               "l2": "not flushed: every step streams the 1.1 GB K/V cache, far above L2"}
    check_device_error(db, "the timed steps")

    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded; shapes of the workload)",
        "config": {"workload": w.name, "B": w.B, "N": w.N, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                   "prefix_len": int(inp.vc.max()), "page_size": w.page_size, "parallelism": f"replicas x{world}",
                   "l2": "flushed before every timed step (512 MiB write, outside the step's events)",
                   "host": f"runs ahead of the device: a GPU spin outside the events before every {AHEAD_STEPS} "
                           "steps lets the host enqueue them, so the device times are the kernels' own"},
        "roofline": roof,
        "verify_tree_us": time_walk(db, stream, args),
        "kernels_us": {n: statistics.median(v) * 1e3 for n, v in per_call.items()},
        "gpu_launches": launches_per_step * args.steps,
        "wall_s_timed_region": wall,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_argmax:
        line["target_argmax"] = time_target_argmax(inp, db, stream, flush, args, hbm)
    if not args.no_lanes:
        line["lane_attention"] = time_lane_attention(stream, flush, args, hbm, tf_sus, db.device)
    if not args.no_fp8:
        line["fp8_attention"] = time_fp8_attention(inp, db, stream, flush, args, hbm, tf_sus)
    if not args.no_side_workloads:
        line["workloads"] = {}
        for name in SIDE_WORKLOADS:
            if name != w.name:
                line["workloads"][name] = time_side_workload(name, args, dev, stream, flush)
    clocks = clk.summary()
    if clocks is not None:
        line["clocks"] = clocks
    if rank == 0 and not args.no_cpu_baseline:
        # about 12 s of oracle work on the host cores
        v, dt, sample = cpu_rows_per_s(inp, steps=1, min_seconds=12.0)
        line["cpu_baseline"] = {"value": v, "unit": "rows/s", "cores": blas_threads(), "kind": "oracle",
                                "sample": sample, "seconds": dt}
    return line


SIDE_WORKLOADS = ("longctx_p131072_n64", "highconc_b128_n16")


def time_side_workload(name, args, dev, stream, flush):
    """One more workload's verify step, timed in the same run as the headline:
    per-call CUDA events over `reps` steps, L2 flushed before each step. The
    attention call gets its roofline (HBM or sustained tensor, whichever
    bounds it). A workload with fp8 layers (the high-concurrency batch) runs
    the full verify step: mask, window K/V, attention, the target argmax over
    its fp32 logits fed straight into the walk (dts_verify_tree_greedy_logits),
    then the compaction of every K/V buffer (the attention layer's bf16 K and V
    plus 2 x fp8_layers fp8 buffers) and of the hidden rows."""
    import torch
    from draft_tree_speculative_gb300 import target_argmax, target_argmax_workspace
    from draft_tree_speculative_gb300.step import DeviceBatch
    w = synth.WORKLOADS[name]
    inp = synth.make_inputs(w)
    db = DeviceBatch(inp, device=dev)
    full = w.fp8_layers > 0
    names = ["prologue", "attention", "epilogue"]
    calls = [db.prologue_step, db.attention_step, db.epilogue_step]
    logits = ws = arg = None
    if full:
        logits = torch.from_numpy(synth.target_logits(w, inp.target_argmax)).to(dev)
        arg = torch.empty((w.B, w.N), dtype=torch.int32, device=dev)
        ws = torch.empty(max(8, target_argmax_workspace(w.B * w.N, w.vocab)), dtype=torch.uint8, device=dev)
        names = ["prologue", "attention", "target_argmax", "epilogue"]
        calls = [db.prologue_step, db.attention_step,
                 lambda st: target_argmax(logits, arg.view(-1), ws, stream=st),
                 lambda st: db.epilogue_step(st, target_argmax=arg)]
    reps = max(5, min(args.steps, 30))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(reps)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            flush.fill_(1)
            for c in calls:
                c(stream)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        with torch.cuda.stream(stream):
            for r, e in enumerate(ev):
                if r % AHEAD_STEPS == 0:
                    run_ahead(stream)
                flush.fill_(1)
                for k, c in enumerate(calls):
                    e[k].record(stream)
                    c(stream)
                e[-1].record(stream)
        torch.cuda.synchronize()
    check_device_error(db, f"the {name} steps")
    per = {n: [e[k].elapsed_time(e[k + 1]) for e in ev] for k, n in enumerate(names)}
    step_us = statistics.median(e[0].elapsed_time(e[-1]) for e in ev) * 1e3
    attn_ms = statistics.mean(per["attention"])
    roof = attention_roofline(inp, attn_ms, name)
    out = {"B": w.B, "N": w.N, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "prefix_len_max": int(inp.vc.max()),
           "prefix_len_sum": int(inp.vc.sum()), "reps": reps,
           "attention_us": attn_ms * 1e3, "rows_per_s": w.B * w.N / (attn_ms / 1e3), "roofline": roof,
           "kernels_us": {n: statistics.median(v) * 1e3 for n, v in per.items()}}
    clocks = clk.summary()
    if clocks is not None:
        out["clocks"] = clocks
    if full:
        out["full_step_us"] = step_us
        out["full_step"] = ("prologue (mask + window K/V), attention, target argmax over fp32 logits "
                            f"[{w.B * w.N}][{w.vocab}], epilogue (walk + compaction of {len(db.kv_entries)} K/V "
                            f"buffers ({2 * w.fp8_layers} fp8 layers' K and V plus the bf16 attention layer) and "
                            f"hidden rows [{w.B * w.N}][{inp.hidden.shape[1]}])")
        out["argmax_matches_planted_target"] = bool((arg.cpu().numpy() == inp.target_argmax).all())
    else:
        out["step_us"] = step_us
    del db, logits, ws, arg
    torch.cuda.empty_cache()
    return out


def time_walk(db, stream, args):
    """verify_tree_greedy alone (the walk over the step's links), CUDA-event
    time per call; in the step it runs inside the fused epilogue."""
    import torch
    reps = max(5, min(args.steps, 50))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            db.walk_step(stream)
        for r, (a, b) in enumerate(ev):
            if r % AHEAD_STEPS == 0:
                run_ahead(stream, 500.0)
            a.record(stream)
            db.walk_step(stream)
            b.record(stream)
    torch.cuda.synchronize()
    check_device_error(db, "the walk")
    return statistics.median(x.elapsed_time(y) for x, y in ev) * 1e3


def time_target_argmax(inp, db, stream, flush, args, hbm):
    """The target's argmax over the workload's fp32 logits [B*N][vocab] and the
    walk fed by it (dts_verify_tree_greedy_logits), outside the headline step:
    CUDA-event time of the argmax call alone and of the fused call, L2 flushed
    before each; the argmax streams the logits once, so its roofline is HBM."""
    import torch
    from draft_tree_speculative_gb300 import (sample_draws, target_argmax, target_argmax_workspace,
                                              verify_tree_greedy_logits, verify_tree_sampled)
    w = inp.w
    rows = w.B * w.N
    logits = torch.from_numpy(synth.target_logits(w, inp.target_argmax)).to(db.device)
    arg = torch.empty((w.B, w.N), dtype=torch.int32, device=db.device)
    ws = torch.empty(max(8, target_argmax_workspace(rows, w.vocab)), dtype=torch.uint8, device=db.device)
    reps = max(5, min(args.steps, 50))

    def timed(fn):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            for a, b in ev:
                flush.fill_(1)
                a.record(stream)
                fn()
                b.record(stream)
        torch.cuda.synchronize()
        return statistics.median(x.elapsed_time(y) for x, y in ev) * 1e3

    us = timed(lambda: target_argmax(logits, arg.view(-1), ws, stream=stream))
    fused_us = timed(lambda: verify_tree_greedy_logits(db.draft, logits, arg, db.accept_len, db.accepted_path,
                                                       db.accepted_tokens, ws, parents=db.parents, err=db.err,
                                                       stream=stream))
    check_device_error(db, "the argmax and walk")
    ok = bool((arg.cpu().numpy() == inp.target_argmax).all())
    nbytes = rows * w.vocab * 4
    gbs = nbytes / (us / 1e6) / 1e9
    # sampled verify (Gumbel-max keyed by position) over the same logits, T = 1
    temp = torch.ones(w.B, dtype=torch.float32, device=db.device)
    seed = torch.arange(w.B, dtype=torch.int64, device=db.device) * 7919 + 1
    draws = torch.empty((w.B, w.N), dtype=torch.int32, device=db.device)
    samp_us = timed(lambda: sample_draws(logits, db.vc, db.depth, temp, seed, draws, ws, stream=stream))
    samp_walk_us = timed(lambda: verify_tree_sampled(db.draft, logits, db.vc, db.depth, temp, seed, draws,
                                                     db.accept_len, db.accepted_path, db.accepted_tokens, ws,
                                                     parents=db.parents, err=db.err, stream=stream))
    check_device_error(db, "the sampled draws and walk")
    elems = rows * w.vocab
    # the sampled draws are bound by instruction issue: achieved warp
    # instructions per second (the profiled count per call, while the source
    # is unchanged) against 4 per SM per cycle at the maximum SM clock
    sm_count = torch.cuda.get_device_properties(db.device).multi_processor_count
    alu_peak = sm_count * 4 * load_sm_max_mhz() * 1e6
    inst = recorded_instructions("sampled_draws", w.name)
    alu = None
    if inst is not None:
        alu = {"bound": "alu", "achieved": inst / (samp_us / 1e6), "peak": alu_peak, "unit": "warp-inst/s",
               "frac": inst / (samp_us / 1e6) / alu_peak, "warp_instructions_per_call": inst}
    return {"us": us, "fused_walk_us": fused_us, "rows": rows, "vocab": w.vocab, "bytes": nbytes,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm},
            "argmax_matches_planted_target": ok, "reps": reps,
            "sampled": {"us": samp_us, "fused_walk_us": samp_walk_us, "logits_per_s": elems / (samp_us / 1e6),
                        "hbm_gbs": nbytes / (samp_us / 1e6) / 1e9, "hbm_frac": nbytes / (samp_us / 1e6) / 1e9 / hbm,
                        "roofline": alu}}


LANE_WORKLOAD = "lanes_eagle2_p8192_k8_s7"


def time_lane_attention(stream, flush, args, hbm, tf_sus, device):
    """Draft-lane attention (dts_tree_window_attention with R = K lane rows
    over the (S - 1) * K-key lane window) on the EAGLE-2 batch's drafting
    shape, outside the headline step: CUDA-event time per call, L2 flushed
    before each; roofline as for the verify attention (K/V of every prefix and
    window key read once per KV head, plus q and out)."""
    import torch
    from draft_tree_speculative_gb300 import tree_window_attention, tree_window_attention_workspace
    lw = synth.LANE_WORKLOADS[LANE_WORKLOAD]
    li = synth.make_lane_inputs(lw)
    B, R, W = lw.B, lw.R, lw.W
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
    q, kc, vc = bf(li.q), bf(li.k_cache), bf(li.v_cache)
    pt, plen, pos = t(li.layout.page_table), t(li.prefix_len), t(li.positions)
    mask = t(li.mask.view(np.int64))
    out = torch.empty((B * R, lw.Hq, lw.d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((B * R, lw.Hq), dtype=torch.float32, device=device)
    max_prefix = int(max(lw.prefix))
    ws = torch.empty(tree_window_attention_workspace(B, R, W, lw.Hq, lw.Hkv, lw.d, max_prefix), dtype=torch.uint8,
                     device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    reps = max(5, min(args.steps, 50))
    call = lambda: tree_window_attention(q, kc, vc, pt, lw.page_size, plen, max_prefix, mask, pos, lw.rope_theta,
                                         out, lse, ws, W, err=err, stream=stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
        for a, b in ev:
            flush.fill_(1)
            a.record(stream)
            call()
            b.record(stream)
    torch.cuda.synchronize()
    if int(err.item()):
        raise RuntimeError(f"device reported error {int(err.item())} in the lane attention")
    us = statistics.median(x.elapsed_time(y) for x, y in ev) * 1e3
    P = np.asarray(lw.prefix, np.int64)
    kv = 2 * lw.Hkv * lw.d * 2 * (int(P.sum()) + B * W)
    rows = B * R * lw.Hq
    nbytes = kv + 2 * rows * lw.d * 2 + rows * 4 + B * R * (8 + 4) + li.layout.page_table.size * 4 + B * 4
    flops = 4 * R * lw.Hq * lw.d * int(P.sum())
    t_hbm, t_mma = nbytes / (hbm * 1e9), flops / (tf_sus * 1e12)
    gbs = nbytes / (us / 1e6) / 1e9
    return {"workload": lw.name, "B": B, "R": R, "W": W, "prefix_len": int(P.max()), "us": us,
            "rows_per_s": B * R / (us / 1e6), "bytes": nbytes, "flops": flops,
            "roofline": {"bound": "hbm" if t_hbm >= t_mma else "tensor", "achieved": gbs, "peak": hbm,
                         "unit": "GB/s", "frac": gbs / hbm}, "reps": reps}


def time_fp8_attention(inp, db, stream, flush, args, hbm, tf_sus):
    """tree_verify_attention_fp8 on the bench workload's shape with unscaled
    E4M3 K/V caches (seeded, N(0,1)-shaped), outside the headline step:
    CUDA-event time per call, L2 flushed before each. The step's own mask,
    positions and queries are reused. Roofline as for the bf16 call with one
    byte per K/V element."""
    import torch
    from draft_tree_speculative_gb300 import tree_verify_attention_fp8
    w = inp.w
    k8, v8 = synth.fp8_kv_cache(w.index, inp.layout.num_slots, w.Hkv, w.d)
    kc, vc = torch.from_numpy(k8).to(db.device), torch.from_numpy(v8).to(db.device)
    del k8, v8
    BN = w.B * w.N
    out = torch.empty((BN, w.Hq, w.d), dtype=torch.bfloat16, device=db.device)
    lse = torch.empty((BN, w.Hq), dtype=torch.float32, device=db.device)
    err = torch.zeros(1, dtype=torch.int32, device=db.device)
    reps = max(5, min(args.steps, 50))
    call = lambda: tree_verify_attention_fp8(db.q, kc, vc, db.page_table, w.page_size, db.prefix_len, db.max_prefix,
                                             db.mask, db.positions, w.rope_theta, out, lse, db.workspace, err=err,
                                             stream=stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            call()
        for a, b in ev:
            flush.fill_(1)
            a.record(stream)
            call()
            b.record(stream)
    torch.cuda.synchronize()
    if int(err.item()):
        raise RuntimeError(f"device reported error {int(err.item())} in the FP8 attention")
    us = statistics.median(x.elapsed_time(y) for x, y in ev) * 1e3
    P = inp.vc.astype(np.int64)
    kv = 2 * w.Hkv * w.d * 1 * (int(P.sum()) + BN)
    rows = BN * w.Hq
    nbytes = kv + 2 * rows * w.d * 2 + rows * 4 + BN * (8 + 4) + inp.layout.page_table.size * 4 + w.B * 4
    flops = 4 * w.N * w.Hq * w.d * int(P.sum())
    # half the flops (S = Q K^T) run as E4M3 MMAs, at twice the measured bf16
    # rate (the nominal fp8 / bf16 ratio); the other half (P V) in f16
    t_hbm = nbytes / (hbm * 1e9)
    t_mma = (flops / 2) / (2 * tf_sus * 1e12) + (flops / 2) / (tf_sus * 1e12)
    t = us / 1e6
    if t_hbm >= t_mma:
        roof = {"bound": "hbm", "achieved": nbytes / t / 1e9, "peak": hbm, "unit": "GB/s", "frac": t_hbm / t}
    else:
        roof = {"bound": "tensor", "achieved": flops / t / 1e12, "peak": flops / t_mma / 1e12, "unit": "TFLOP/s",
                "frac": t_mma / t,
                "peak_source": "measured sustained bf16 x 2 for the E4M3 half (S), x 1 for the f16 half (P V)"}
    roof["hbm_frac"] = t_hbm / t
    roof["traffic_tree_pass"] = recorded_traffic("fp8:" + w.name)
    return {"workload": w.name, "kv_dtype": "e4m3 (unscaled)",
            "compute": ("prefix keys: E4M3 S MMA (query cast to E4M3), f16 P V MMA (V widened), fp32 accumulation; "
                        "window keys: bf16 query against exactly widened E4M3 K/V in fp32; parts merged by LSE"),
            "us": us, "rows_per_s": BN / t, "bytes": nbytes, "flops": flops, "roofline": roof, "reps": reps}


def run_reference(args):
    w = synth.WORKLOADS[args.workload]
    inp = synth.make_inputs(w)
    cpu_rows_per_s(inp, steps=args.warmup)
    v, dt, sample = cpu_rows_per_s(inp, steps=args.steps)
    line = {
        "metric": METRIC, "value": v, "unit": "rows/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; shapes of the workload)",
        "config": {"workload": w.name, "B": w.B, "N": w.N, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d,
                   "prefix_len": int(inp.vc.max()), "page_size": w.page_size, "parallelism": "host cores"},
        "impl": "reference",
        "cpu_baseline": {"value": v, "unit": "rows/s", "cores": blas_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)))
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
