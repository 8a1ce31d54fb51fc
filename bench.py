"""Benchmark of the Multi-Segment Attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl msa|reference] [--quick]

One step = one pass of the hot path over one batch: the step's new K/V
appended into the paged pool (msa_append_kv) and attention of every query
row over all segments of all sequences in one persistent launch
(msa_attention).  The plan (segments + balanced work list) is built once per
batch on the host and uploaded before the timed region; its host cost is
reported as plan_us.  The K timed steps are issued back to back with CUDA
events at their ends only; the attention kernel's own duration (the
roofline's denominator) comes from a second pass of K steps with an event
pair around each attention launch.  The e2e figure rebuilds and uploads the plan from host
arrays every step and copies the step's inputs/outputs through pinned host
memory.

Headline workload: batched decode, Llama-3-8B attention shape (32 sequences,
32/8 heads, D=128, contexts U{2k..16k}, 1-8 segments each, in a 4M-token
pool).  Metric: decode HBM GB/s of algorithmic bytes (K+V of every visible
key once, q, out, lse, plus the append's bytes).  Extra lines in the same
JSON object: hole-recompute prefill TFLOP/s, long-context and mixed-batch
runs, and the segmented-vs-contiguous overhead.

Prints ONE JSON line (rank 0).  Under torchrun each rank runs its own batch
(different seed, same shape): weak scaling, no data-path collective; the
value is the sum of all ranks' bytes over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MSA attention: decode HBM GB/s, prefill TFLOP/s (% of GB300 roofline)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def code_sha(path):
    """First 12 hex digits of the sha1 of a source file's code: comments
    removed and whitespace runs folded, so that a capture stays valid across
    edits of comments only."""
    import hashlib
    import re
    src = open(path, encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    src = re.sub(r"\s+", " ", src)
    return hashlib.sha1(src.encode()).hexdigest()[:12]


def load_traffic():
    """Per-launch DRAM bytes from the committed ncu summaries (profiles/*.txt
    lines `traffic <workload> <bytes> <source-sha>`), kept only while the
    kernel source is unchanged."""
    src = os.path.join(ROOT, "kv_cache_segment_gb300", "csrc", "attention.cu")
    sha = code_sha(src) if os.path.exists(src) else ""
    out = {}
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return out
    for f in sorted(os.listdir(pdir)):
        if not f.endswith(".txt"):
            continue
        for line in open(os.path.join(pdir, f)):
            parts = line.split()
            if len(parts) == 4 and parts[0] == "traffic" and parts[3] == sha:
                out[parts[1]] = float(parts[2])
    return out


# ------------------------------------------------------------- clocks --

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None, interval_ms=50):
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", str(interval_ms)]
        if gpu_id:
            cmd[1:1] = ["-i", gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for t, line in self.samples:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((t, parts))
        # samples inside the timed region; if it was shorter than the sampling
        # interval, the ones closest to it (within 0.25 s)
        inside = [r for r in rows if self.t0 is not None and self.t0 <= r[0] <= (self.t1 or r[0])]
        if not inside:
            inside = [r for r in rows if self.t0 is not None and self.t0 - 0.25 <= r[0] <= (self.t1 or self.t0) + 0.25]
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1][1]) for r in inside if num(r[1][1]) is not None]
        mx = [num(r[1][2]) for r in inside if num(r[1][2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4) if r[1][5 + i].lower().startswith("active")})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside)}


# ------------------------------------------------------------ GPU legs --

class Case:
    """A workload resident on the GPU: pools, q, plan, workspace, outputs."""

    def __init__(self, wl, dev, contiguous=False, plan_opts=None):
        import torch
        from kv_cache_segment_gb300 import msa
        from kv_cache_segment_gb300 import workloads as W
        from kv_cache_segment_gb300.runner import MsaSession
        if contiguous:
            wl = _contiguous_copy(wl)
        self.wl = wl
        self.dev = dev
        k, v, q = W.make_values(wl, device=dev)
        self.kp, self.vp = W.make_pool(wl, k, v, fill=0.0)
        del k, v
        self.q = q
        self.sess = MsaSession.from_workload(wl, device=dev, **(plan_opts or {}))
        self.info = self.sess.info
        self.out = torch.empty((wl.num_q_rows, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((wl.num_q_rows, wl.num_q_heads), dtype=torch.float32, device=dev)
        self.dims = msa.make_dims(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, 16, wl.scale)
        # the step's appended K/V: one new token per decode sequence plus every
        # prefill row's own K/V (recomputed holes / new turn), written to the
        # rows the layout gives them
        slots = wl.slot_mapping()
        rows = []
        kv_ind = wl.kv_indptr
        for s in range(wl.num_seqs):
            for (a, b) in wl.q_ranges[s]:
                hi = min(b, int(wl.seq_lens[s]))
                if hi > a:
                    rows.append(np.arange(kv_ind[s] + a, kv_ind[s] + hi))
        idx = np.concatenate(rows) if rows else np.zeros(0, np.int64)
        n_dec = sum(1 for s in range(wl.num_seqs) for (a, b) in wl.q_ranges[s] if b == int(wl.seq_lens[s]) + 1)
        # decode sequences append their new token into rows of free blocks
        used = np.zeros(wl.pool_blocks, bool)
        used[wl.block_table[wl.block_table >= 0]] = True
        free_blocks = np.flatnonzero(~used)[:n_dec]
        spare = free_blocks.astype(np.int64) * 16
        self.slot = torch.from_numpy(np.concatenate([slots[idx], spare]).astype(np.int64)).to(dev)
        n_new = len(self.slot)
        g = torch.Generator(device=dev)
        g.manual_seed(wl.seed + 17)
        self.k_new = torch.randn((n_new, wl.num_kv_heads, wl.head_dim), generator=g, device=dev).to(torch.bfloat16)
        self.v_new = torch.randn((n_new, wl.num_kv_heads, wl.head_dim), generator=g, device=dev).to(torch.bfloat16)
        if len(idx):
            # the recomputed rows equal what the pool already holds for them
            sl = torch.from_numpy(slots[idx].astype(np.int64)).to(dev)
            self.k_new[: len(idx)] = self.kp[sl]
            self.v_new[: len(idx)] = self.vp[sl]
        self.append_bytes = 2 * 2 * n_new * wl.num_kv_heads * wl.head_dim * 2 + n_new * 8
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)

    def append(self, stream):
        from kv_cache_segment_gb300 import msa
        if len(self.slot):
            msa.msa_append_kv(self.k_new, self.v_new, self.slot, len(self.slot), self.kp, self.vp,
                              self.kp.shape[0], self.dims, self.err, stream)

    def attention(self, stream):
        from kv_cache_segment_gb300 import msa
        msa.msa_attention(self.q, self.kp, self.vp, self.kp.shape[0], self.sess.plan, self.out, msa.MSA_OUT_BF16,
                          self.lse, stream)

    def replan(self, **plan_opts):
        """Replace the session's plan (same workload) by one made with other
        msa_plan_create_ex options."""
        from kv_cache_segment_gb300.runner import MsaSession
        self.sess.close()
        self.sess = MsaSession.from_workload(self.wl, device=self.dev, **plan_opts)
        self.info = self.sess.info

    def decode_bytes(self):
        return self.info["decode_kv_bytes"] + self.info["decode_qo_bytes"]

    def flops(self):
        return self.info["prefill_flops"]


def _contiguous_copy(wl):
    """Same sequences and queries, each sequence stored as one run."""
    from kv_cache_segment_gb300 import workloads as W
    lay = W._Layout(wl.num_seqs)
    for s in range(wl.num_seqs):
        nb = -(-int(wl.seq_lens[s]) // 16)
        if nb:
            lay.run(s, nb)
    rng = np.random.default_rng(wl.seed + 99)
    return W._finish(wl.name + "_contiguous", wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.seq_lens, lay,
                     wl.pool_blocks, wl.q_ranges, rng, wl.seed)


def time_case(case, steps, warmup, stream, with_append=True):
    """Per-step device time (ms) of [append +] attention, and the attention
    kernel's own average duration, CUDA events on the launching stream."""
    import torch
    for _ in range(warmup):
        if with_append:
            case.append(stream)
        case.attention(stream)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for e in ev:
        e[0].record(stream)
        if with_append:
            case.append(stream)
        e[1].record(stream)
        case.attention(stream)
        e[2].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    total = start.elapsed_time(end)
    attn = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
    return total / steps, attn


def gpu_main(args):
    import torch
    import torch.distributed as dist
    from kv_cache_segment_gb300 import msa
    from kv_cache_segment_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus > 1 and world == 1:
        print(json.dumps({"error": "use torchrun for --gpus > 1"}))
        return 2
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        try:
            dist.init_process_group("nccl", device_id=dev)
        except TypeError:
            dist.init_process_group("nccl")
    msa.load()
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream(dev)

    # ---- headline: batched decode -------------------------------------
    wl = W.config(2, seed=1002 + 1000 * rank)
    case = Case(wl, dev, plan_opts=_plan_opts())
    step_bytes = case.decode_bytes() + case.append_bytes
    gpu_id = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        gpu_id = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)
    for _ in range(args.warmup):
        case.append(stream)
        case.attention(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # The timed steps: append + attention back to back, as a serving loop
    # issues them (the attention launch overlaps the append's end through
    # programmatic dependent launch, which an event recorded between the two
    # would stop), events only at the ends.
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    sampler.mark_start()
    t_start.record(stream)
    for _ in range(args.steps):
        case.append(stream)
        case.attention(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    sampler.mark_end()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    elapsed_ms = t_start.elapsed_time(t_end)
    # The attention kernel's own duration for the roofline: the same K steps
    # again with an event pair around each attention launch.
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for e in ev:
        case.append(stream)
        e[0].record(stream)
        case.attention(stream)
        e[1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    attn_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    rc, word = case.sess.check_device()
    if rc != 0 or int(case.err.item()) != 0:
        raise RuntimeError(f"device error word {word:#x} / append {int(case.err.item())}")
    elapsed_ms, total_bytes = reduce_over_ranks(elapsed_ms, step_bytes, dev if world > 1 else None)
    ms_per_step = elapsed_ms / args.steps
    value = total_bytes / (ms_per_step * 1e-3) / 1e9

    traffic = load_traffic()
    attn_bytes = case.decode_bytes()
    achieved = attn_bytes / (attn_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": f"{peak_src} (hbm_gbs, of {peak_src})",
                "kernel": "msa_attention_kernel<128>", "algorithmic_bytes_per_launch": attn_bytes,
                "kernel_ms": round(attn_ms, 5),
                "kernel_ms_source": "CUDA events around each attention launch, a second pass of the K steps",
                "traffic": traffic.get("batched_decode")}

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "batched_decode: 32 seqs x 1 decode row, 32/8 heads, D=128, block 16, "
                               "L~U{2048..16384}, 1-8 segments/seq in a 4M-token pool",
                   "seqs_per_gpu": wl.num_seqs, "segments": int(case.info["num_runs"]),
                   "items": int(case.info["num_items"]), "grid": int(case.info["grid"]),
                   "kv_bytes_per_step": int(case.info["decode_kv_bytes"]),
                   "l2": "inputs larger than L2 (K/V read per step >> 129 MB L2; 16 GiB pools)",
                   "planner": _planner_note(case),
                   "parallelism": f"replicas x{world} (independent batches, no collective)"},
        "roofline": roofline,
        "plan_us": round(case.info["host_plan_us"], 1),
        "clocks": clocks,
        "gpu_launches": 2 * args.steps,
    }

    headline_pred = _predict_us(case)
    if rank == 0 and not args.quick:
        result["e2e"] = e2e_leg(case, args, dev, stream)
    del case
    torch.cuda.empty_cache()

    if not args.quick:
        extras = extra_legs(args, dev, stream, peaks, peak_src, traffic, rank)
        if "cost_model" in extras and headline_pred is not None:
            m = attn_ms * 1e3
            extras["cost_model"]["batched_decode"] = {"predicted_us": headline_pred, "measured_us": round(m, 1),
                                                      "rel_err": round(headline_pred / m - 1.0, 4)}
        result.update(extras)
    if world > 1:
        dist.barrier()
    if rank == 0:
        if not args.quick and not args.no_cpu:
            result["cpu_baseline"] = cpu_baseline(wl, target_s=args.cpu_seconds)
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def reduce_over_ranks(elapsed_ms, nbytes, device=None):
    """Whole-job figures: the slowest rank's time and the sum of all ranks'
    bytes (no-op without an initialised process group)."""
    import torch
    import torch.distributed as dist
    if device is None or not (dist.is_available() and dist.is_initialized()):
        return float(elapsed_ms), float(nbytes)
    t = torch.tensor([float(elapsed_ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    b = torch.tensor([float(nbytes)], device=device, dtype=torch.float64)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


def e2e_leg(case, args, dev, stream):
    """Same metric through the C ABI from host buffers.  Every step: the plan
    is built from the host block tables and uploaded, q and the new K/V go
    up from pinned memory, append + attention run, out and lse come back to
    pinned memory and the host reads them.  As a serving loop would, the
    steps are pipelined two deep (the host builds and issues step i+1 before
    it waits for step i's results) with two sets of device buffers and
    workspaces taking turns, and the copies run on two copy streams: step
    i+1's inputs go up while step i computes, and step i's results come back
    while step i+1 computes.  Events order each buffer set's uses: a set's
    inputs are overwritten only after the attention two steps back has read
    them, and its output only after the copy of that step's results is done.
    The inputs of a step travel as one packed pinned buffer (q | K new | V
    new | slots) and the results as one (out | lse)."""
    import torch
    from kv_cache_segment_gb300 import msa
    wl = case.wl
    parts_in = [case.q, case.k_new, case.v_new, case.slot]
    parts_out = [case.out, case.lse]

    def layout(parts):
        offs, o = [], 0
        for t in parts:
            offs.append(o)
            o += -(-t.numel() * t.element_size() // 16) * 16  # 16-byte aligned pieces
        return offs, o

    in_off, in_bytes = layout(parts_in)
    out_off, out_bytes = layout(parts_out)

    def views(buf, parts, offs):
        return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for t, o in zip(parts, offs)]

    in_h = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    for v, t in zip(views(in_h, parts_in, in_off), parts_in):
        v.copy_(t.cpu())
    two = lambda f: [f(), f()]  # noqa: E731
    in_d = two(lambda: torch.empty(in_bytes, dtype=torch.uint8, device=dev))
    out_d = two(lambda: torch.empty(out_bytes, dtype=torch.uint8, device=dev))
    out_h = two(lambda: torch.empty(out_bytes, dtype=torch.uint8).pin_memory())
    vin = [views(b, parts_in, in_off) for b in in_d]    # [q, k_new, v_new, slot] per set
    vout = [views(b, parts_out, out_off) for b in out_d]  # [out, lse] per set
    lse_h = [views(b, parts_out, out_off)[1] for b in out_h]
    ws = [case.sess.workspace, torch.empty_like(case.sess.workspace)]
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in, ev_attn, ev_out = two(torch.cuda.Event), two(torch.cuda.Event), two(torch.cuda.Event)
    table, lens = wl.block_table, wl.seq_lens
    indptr, ranges = wl.q_range_indptr, wl.q_ranges_flat
    n_new = len(case.slot)
    dsplit, psplit, grid = case.info["decode_split"], case.info["prefill_split"], case.info["grid"]
    check = [0.0]
    host_s = [0.0]

    def issue(i):
        """Plan, upload and launch step i on buffer set i % 2; returns (plan,
        plan bytes)."""
        t0 = time.perf_counter()
        b = i % 2
        # the split factors the session's plan was chosen with, reused: a
        # planner call per step stays as cheap as the default one
        plan = msa.msa_plan_create_ex(case.dims, table, lens, indptr, ranges, grid, dsplit, psplit)
        nbytes = msa.msa_plan_workspace_bytes(plan)
        if nbytes > ws[b].numel():
            raise RuntimeError("per-step plan larger than the session's workspace")
        h2d_s.wait_event(ev_attn[b])  # set b's inputs and workspace were read by step i-2
        msa.msa_plan_upload(plan, ws[b], nbytes, h2d_s)
        with torch.cuda.stream(h2d_s):
            in_d[b].copy_(in_h, non_blocking=True)
        ev_in[b].record(h2d_s)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])  # step i-2's results have left set b's output
        q_d, kn_d, vn_d, slot_d = vin[b]
        o_d, l_d = vout[b]
        msa.msa_append_kv(kn_d, vn_d, slot_d, n_new, case.kp, case.vp, case.kp.shape[0], case.dims, case.err, stream)
        msa.msa_attention(q_d, case.kp, case.vp, case.kp.shape[0], plan, o_d, msa.MSA_OUT_BF16, l_d, stream)
        ev_attn[b].record(stream)
        d2h_s.wait_event(ev_attn[b])
        with torch.cuda.stream(d2h_s):
            out_h[b].copy_(out_d[b], non_blocking=True)
        ev_out[b].record(d2h_s)
        host_s[0] += time.perf_counter() - t0
        return plan, nbytes

    def finish(i, step):
        plan, _ = step
        ev_out[i % 2].synchronize()  # step i's results are in host memory
        check[0] += float(lse_h[i % 2][0, 0])  # the host reads them
        msa.msa_plan_destroy(plan)

    def run(n_steps):
        prev = issue(0)
        nbytes = prev[1]
        for i in range(1, n_steps):
            cur = issue(i)  # step i is issued before step i-1 is waited for
            finish(i - 1, prev)
            prev = cur
        finish(n_steps - 1, prev)
        return nbytes

    run(max(3, args.warmup))
    torch.cuda.synchronize()
    host_s[0] = 0.0
    t0 = time.perf_counter()
    plan_bytes = run(args.steps)
    dt = (time.perf_counter() - t0) / args.steps
    torch.cuda.synchronize()
    # restore the session's own plan in its workspace
    msa.msa_plan_upload(case.sess.plan, ws[0], case.sess.ws_bytes, stream)
    torch.cuda.synchronize()
    if not math.isfinite(check[0]):
        raise RuntimeError("e2e leg read a non-finite lse")
    # the last step's results, read back through the pipeline, are the bits
    # the device-timed path computes with the same plan (the kernel is
    # deterministic for a plan; the appended rows are the same every step)
    case.append(stream)
    case.attention(stream)
    torch.cuda.synchronize()
    o_h, l_h = views(out_h[(args.steps - 1) % 2], parts_out, out_off)
    if not (torch.equal(o_h.view(torch.int16), case.out.cpu().view(torch.int16))
            and torch.equal(l_h, case.lse.cpu())):
        raise RuntimeError("e2e leg results differ from the device path's")
    val = (case.decode_bytes() + case.append_bytes) / dt / 1e9
    h2d = sum(t.numel() * t.element_size() for t in parts_in)
    d2h = sum(t.numel() * t.element_size() for t in parts_out)
    return {"value": round(val, 1), "unit": "GB/s", "ms_per_step": round(dt * 1e3, 4),
            "h2d_bytes_per_step": int(h2d + plan_bytes), "d2h_bytes_per_step": int(d2h),
            "host_issue_us_per_step": round(host_s[0] / args.steps * 1e6, 1),
            "note": "per step: plan from host block tables (msa_plan_create_ex with the session's split factors) "
                    "uploaded, inputs up from pinned memory, append + attention, out + lse back to pinned "
                    "memory and read by the host; steps pipelined two deep (step i+1 issued before step i "
                    "is waited for), copies on two copy streams overlapping the neighbouring steps' kernels; the last "
                    "step's out and lse equal the device path's bit for bit"}


def _plan_opts():
    """Plans made by msa_plan_create_ex with the adaptive-chunking chooser
    (latency-model constants fitted on this GPU), or the default plan when
    no fit is stored."""
    from kv_cache_segment_gb300 import costfit
    params = costfit.load_params()
    return {"choose_with": params} if params is not None else {}


def _planner_note(case):
    return {"decode_split": case.info["decode_split"], "prefill_split": case.info["prefill_split"],
            "chosen_by": "latency model (msa_plan_create_ex)" if _plan_opts() else "defaults"}


def _predict_us(case):
    """msa_plan_estimate of the case's plan under the fitted constants, or None."""
    from kv_cache_segment_gb300 import costfit, msa
    params = costfit.load_params()
    if params is None:
        return None
    return round(msa.msa_plan_estimate(case.sess.plan, params)["time_us"], 1)


def gather_leg(case, steps, warm, stream):
    """The path MSA replaces (AsymCache explainer, "核心方法 1"): gather the
    batch's scattered K/V into one contiguous, block-aligned buffer
    (msa_gather_kv), then attention over that buffer with one segment per
    sequence; against msa_attention on the segmented layout.  Device time per
    step, CUDA events on the launching stream."""
    import dataclasses
    import torch
    from kv_cache_segment_gb300 import msa
    from kv_cache_segment_gb300.runner import MsaSession
    wl = case.wl
    nb = [-(-int(L) // 16) for L in wl.seq_lens]
    base = np.concatenate([[0], np.cumsum(nb)]).astype(np.int64)
    rows = int(base[-1]) * 16
    src = np.full(rows, -1, np.int64)
    seg_slots = wl.slot_mapping()
    ind = wl.kv_indptr
    table = np.full((wl.num_seqs, max(1, max(nb) if nb else 1)), -1, np.int32)
    for s in range(wl.num_seqs):
        L = int(wl.seq_lens[s])
        src[base[s] * 16: base[s] * 16 + L] = seg_slots[ind[s]:ind[s] + L]
        table[s, :nb[s]] = base[s] + np.arange(nb[s])
    cont = dataclasses.replace(wl, block_table=table, pool_blocks=max(1, int(base[-1])),
                               runs_drawn=[[(0, int(base[s]), nb[s])] for s in range(wl.num_seqs)],
                               name=wl.name + "/gathered")
    sess = MsaSession.from_workload(cont, device=case.dev, **_plan_opts())
    shape = (max(rows, 1), wl.num_kv_heads, wl.head_dim)
    kg = torch.empty(shape, dtype=torch.bfloat16, device=case.dev)
    vg = torch.empty(shape, dtype=torch.bfloat16, device=case.dev)
    src_d = torch.from_numpy(src).to(case.dev)
    err = torch.zeros(1, dtype=torch.int32, device=case.dev)

    def gather():
        msa.msa_gather_kv(case.kp, case.vp, case.kp.shape[0], src_d, rows, kg, vg, case.dims, err, stream)

    def attend():
        msa.msa_attention(case.q, kg, vg, rows, sess.plan, case.out, msa.MSA_OUT_BF16, case.lse, stream)

    def timed(fns):
        for _ in range(warm):
            for f in fns:
                f()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            for f in fns:
                f()
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / steps

    g_ms = timed([gather])
    a_ms = timed([attend])
    ga_ms = timed([gather, attend])
    m_ms = timed([lambda: case.attention(stream)])
    rc, word = sess.check_device()
    if rc != 0 or int(err.item()) != 0:
        raise RuntimeError(f"gather leg: device error {word:#x} / {int(err.item())}")
    sess.close()
    return {"msa_ms": round(m_ms, 4), "gather_ms": round(g_ms, 4), "contiguous_attention_ms": round(a_ms, 4),
            "gather_plus_attention_ms": round(ga_ms, 4), "msa_speedup": round(ga_ms / m_ms, 3),
            "gathered_bytes": int(rows * wl.num_kv_heads * wl.head_dim * 2 * 2)}


def eviction_workloads(seed=1100, num_seqs=16, blocks=512, evict=128, hq=32, hkv=8, d=128):
    """Synthetic hit probabilities and the eviction choices of three weightings
    of the kernel-aware score (msa_select_evictions): hit probability only,
    recompute cost only, both; and the expected-cost mode, the set with the
    least expected recompute time (lowest hit probability x cost).  Those use
    the hole reading of the recompute cost (only the evicted block is
    rebuilt); two more policies, cost only and hit and cost, use the prefix
    reading (a block is usable only with its whole prefix, so evicting b
    leaves b .. end to rebuild).  Per policy the recompute workload that
    follows when every evicted block is needed again: hole reading: live
    segments where they were, each evicted hole recomputed into fresh
    blocks, queries = the evicted positions and the decode row; prefix
    reading: the live prefix before the first evicted block, everything from
    there to the end recomputed into one fresh run, queries = those positions
    and the decode row.

    Hit probabilities per block (seeded): attention-sink blocks at the start
    (0.9), a recency ramp over the last blocks (0.85 e^-(age/32)), and a
    sparse background (Beta(0.5, 4)); clipped to [0, 1]."""
    from kv_cache_segment_gb300 import costfit, msa
    from kv_cache_segment_gb300 import workloads as W
    params = costfit.load_params() or dict(launch_us=0.0, dec_item_us=0.0, dec_gbs=6400.0, dec_cta_gbs=60.0,
                                           pre_item_us=30.0, pre_tile_us=0.8, box_us=0.0, dec_merge_us=8.0, pre_merge_us=20.0)
    rng = np.random.default_rng(seed)
    L = blocks * 16
    dims = msa.make_dims(hq, hkv, d)
    hits = []
    for _ in range(num_seqs):
        b = np.arange(blocks)
        p = 0.9 * (b < 4) + 0.85 * np.exp(-(blocks - 1 - b) / 32.0) + rng.beta(0.5, 4.0, blocks)
        hits.append(np.clip(p, 0.0, 1.0).astype(np.float32))
    out = {}
    policies = (("hit_only", (1.0, 0.0), False), ("cost_only", (0.0, 1.0), False),
                ("hit_and_cost", (1.0, 1.0), False), ("expected_cost_optimum", None, False),
                ("prefix_cost_only", (0.0, 1.0), True), ("prefix_hit_and_cost", (1.0, 1.0), True))
    for name, weights, prefix in policies:
        alpha, beta = weights if weights else (None, None)
        runs, ranges = [], []
        exp_hits = exp_flops = exp_us = all_flops = 0.0
        first = []
        for s in range(num_seqs):
            pre = msa.MSA_EVICT_PREFIX_COST if prefix else 0
            if weights:
                ev, cost = msa.msa_select_evictions(dims, L, hits[s], alpha, beta, params, evict, mode=pre)
            else:  # the set with the least expected recompute time
                ev, cost = msa.msa_select_evictions(dims, L, hits[s], 0.0, 0.0, params, evict,
                                                    mode=msa.MSA_EVICT_EXPECTED_COST | pre)
            exp_hits += float(hits[s][ev].sum())
            if prefix:
                # every block from the first evicted one on is rebuilt
                b0 = int(ev.min())
                first.append(b0)
                all_flops += 4.0 * d * hq * sum(range(16 * b0 + 1, L + 1))
                runs.append([b0, blocks - b0] if b0 > 0 else [blocks])
                ranges.append([(16 * b0, L), (L, L + 1)])
                continue
            gone = np.zeros(blocks, bool)
            gone[ev] = True
            exp_us += float((hits[s][ev] * cost[ev]).sum())
            keys = np.array([sum(range(16 * b + 1, 16 * b + 17)) for b in ev], np.float64)
            exp_flops += float((hits[s][ev] * 4.0 * d * hq * keys).sum())
            all_flops += float((4.0 * d * hq * keys).sum())
            sizes, rr = [], []
            b = 0
            while b < blocks:  # alternate live segments and holes, in logical order
                e = b
                while e < blocks and gone[e] == gone[b]:
                    e += 1
                sizes.append(e - b)
                if gone[b]:
                    rr.append((16 * b, 16 * e))
                b = e
            rr.append((L, L + 1))
            runs.append(sizes)
            ranges.append(rr)
        wl = W.custom([L] * num_seqs, runs, ranges, hq=hq, hkv=hkv, d=d, seed=seed, name=f"eviction/{name}")
        ent = {"wl": wl, "alpha": alpha, "beta": beta, "cost_reading": "prefix" if prefix else "hole",
               "expected_hit_blocks": round(exp_hits, 2), "all_hit_recompute_gflop": round(all_flops / 1e9, 3),
               "segments_after_recompute": int(sum(len(r) for r in runs))}
        if prefix:
            ent["first_evicted_block_mean"] = round(float(np.mean(first)), 1)
        else:
            ent["expected_recompute_gflop"] = round(exp_flops / 1e9, 3)
            ent["model_expected_recompute_us"] = round(exp_us, 1)
        out[name] = ent
    return out


def eviction_leg(dev, stream, steps, warm):
    import torch
    res = {}
    for name, ent in eviction_workloads().items():
        wl = ent.pop("wl")
        case = Case(wl, dev, plan_opts=_plan_opts())
        step_ms, attn_ms = time_case(case, steps, warm, stream)
        ent["all_hit_recompute"] = {"step_ms": round(step_ms, 4), "attention_ms": round(attn_ms, 4),
                                    "prefill_tflop": round(case.flops() / 1e12, 3),
                                    "predicted_us": _predict_us(case)}
        res[name] = ent
        del case
        torch.cuda.empty_cache()
    return res


def chunking_leg(dev, stream, steps, warm, budget_us=500.0):
    """Adaptive prefill chunk size on the mixed batch (64 decode rows + 4
    pending prefills of their last <= 8192 positions, 64/8 heads, D=128):
    msa_choose_prefill_chunk's choice, unconstrained and under a step budget,
    against fixed chunks of 512 to 4096; for each, the measured step
    (attention) time, prefill tokens per second and the model's prediction.
    Plans use the default split factors, as the chooser's plans do."""
    import torch
    from kv_cache_segment_gb300 import costfit, msa
    from kv_cache_segment_gb300 import workloads as W
    params = costfit.load_params()
    if params is None:
        return {"skipped": "no fitted latency-model constants"}
    wl = W.config(5)
    base, pending = W.pending_prefills(wl)
    dims = msa.make_dims(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, 16, wl.scale)
    grid = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {"pending": [list(p) for p in pending], "budget_us": budget_us}
    chosen = {}
    for key, b in (("chosen", 0.0), ("chosen_within_budget", budget_us)):
        ch, cands, times = msa.msa_choose_prefill_chunk(dims, base.block_table, base.seq_lens, base.q_range_indptr,
                                                         base.q_ranges_flat, pending, params, budget_us=b,
                                                         num_sms=grid)
        chosen[key] = ch["chunk"]
        out[key] = {"chunk": ch["chunk"], "predicted_us": round(ch["time_us"], 1),
                    "within_budget": bool(ch["within_budget"]), "candidates": int(ch["n_candidates"])}
    rows = {}
    for c in sorted({512, 1024, 2048, 4096, *chosen.values()}):
        step = W.with_prefill_chunk(base, pending, c)
        case = Case(step, dev)
        _, attn_ms = time_case(case, steps, warm, stream, with_append=False)
        tokens = sum(min(c, e - a) for _, a, e in pending)
        rows[str(c)] = {"attention_ms": round(attn_ms, 4), "prefill_tokens": tokens,
                        "prefill_tokens_per_s": round(tokens / (attn_ms * 1e-3), 1),
                        "us_per_token": round(attn_ms * 1e3 / tokens, 4),
                        "predicted_us": _predict_us(case)}
        del case
        torch.cuda.empty_cache()
    out["steps"] = rows
    best = min(rows, key=lambda k: rows[k]["us_per_token"])
    out["best_measured_chunk"] = int(best)
    out["chosen_vs_best_us_per_token"] = round(rows[str(chosen["chosen"])]["us_per_token"] /
                                               rows[best]["us_per_token"], 4)
    return out


def extra_legs(args, dev, stream, peaks, peak_src, traffic, rank):
    """Prefill/recompute TFLOP/s (hole recompute + new turn), long context,
    mixed batch, and segmented vs contiguous layouts."""
    import torch
    from kv_cache_segment_gb300 import workloads as W
    steps = max(3, min(args.steps, 10))
    warm = max(3, min(args.warmup, 5))
    out = {}
    lines = {}
    over = {}
    gathers = {}
    for idx, key in ((3, "hole_recompute"), (4, "long_context"), (5, "mixed_batch"), (2, "batched_decode")):
        wl = W.config(idx, seed=1000 + idx + 1000 * rank)
        case = Case(wl, dev, plan_opts=_plan_opts())
        if key != "batched_decode":
            step_ms, attn_ms = time_case(case, steps, warm, stream)
            fl, by = case.flops(), case.decode_bytes()
            ent = {"ms_per_step": round(step_ms, 4), "attention_ms": round(attn_ms, 4),
                   "prefill_tflops": round(fl / (attn_ms * 1e-3) / 1e12, 2) if fl else 0.0,
                   "decode_kv_gbs_in_mixed_launch": round(by / (attn_ms * 1e-3) / 1e9, 1) if by else 0.0,
                   "items": int(case.info["num_items"]), "segments": int(case.info["num_runs"]),
                   "append_bytes": int(case.append_bytes)}
            if fl:
                ent["tensor_frac"] = round(fl / (attn_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)
            # additive lower bound on time for a mixed launch
            lb = by / (peaks["hbm_gbs"] * 1e9) + fl / (peaks["bf16_tflops"] * 1e12)
            ent["roofline_frac_additive"] = round(lb / (attn_ms * 1e-3), 4)
            ent["traffic"] = traffic.get(key)
            ent["predicted_us"] = _predict_us(case)
            ent["planner"] = _planner_note(case)
            if _plan_opts():
                # the same launch with the default split factors
                case.replan()
                _, def_ms = time_case(case, steps, warm, stream, with_append=False)
                ent["default_plan_attention_ms"] = round(def_ms, 4)
                case.replan(**_plan_opts())
            if key in ("long_context", "mixed_batch"):
                # graded per-kind rates: the same sequences, layout and tiling
                # with only the decode rows, then only the prefill rows
                for kind in ("decode", "prefill"):
                    sub = Case(W.restrict_rows(wl, kind), dev, plan_opts=_plan_opts())
                    _, sub_ms = time_case(sub, steps, warm, stream, with_append=False)
                    if kind == "decode":
                        gbs = sub.decode_bytes() / (sub_ms * 1e-3) / 1e9
                        ent["decode_only"] = {"attention_ms": round(sub_ms, 4), "decode_gbs": round(gbs, 1),
                                              "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                                              "items": int(sub.info["num_items"])}
                    else:
                        tf = sub.flops() / (sub_ms * 1e-3) / 1e12
                        ent["prefill_only"] = {"attention_ms": round(sub_ms, 4), "prefill_tflops": round(tf, 2),
                                               "tensor_frac": round(tf / peaks["bf16_tflops"], 4),
                                               "items": int(sub.info["num_items"])}
                    del sub
                    torch.cuda.empty_cache()
            lines[key] = ent
        if key in ("hole_recompute", "batched_decode", "long_context"):
            gathers[key] = gather_leg(case, steps, warm, stream)
            torch.cuda.empty_cache()
            # the same sequences laid out as one contiguous run each, timed in
            # alternation with the segmented layout (median of three rounds)
            # so that both see the same state of the GPU
            cont = Case(wl, dev, contiguous=True, plan_opts=_plan_opts())
            seg_t, con_t = [], []
            for _ in range(3):
                seg_t.append(time_case(case, steps, warm, stream, with_append=False)[1])
                con_t.append(time_case(cont, steps, warm, stream, with_append=False)[1])
            seg_ms, con_ms = float(np.median(seg_t)), float(np.median(con_t))
            over[key] = {"segmented_ms": round(seg_ms, 4), "contiguous_ms": round(con_ms, 4),
                         "ratio": round(seg_ms / con_ms, 4)}
            del case, cont
        else:
            del case
        torch.cuda.empty_cache()
    # expected-latency model (msa_plan_estimate, constants fitted on this
    # GPU) against the measured launches
    from kv_cache_segment_gb300 import costfit
    params = costfit.load_params()
    if params is not None:
        cm = {}
        for key, ent in lines.items():
            if "predicted_us" in ent:
                cm[key] = {"predicted_us": ent.pop("predicted_us"), "measured_us": round(ent["attention_ms"] * 1e3, 1)}
                cm[key]["rel_err"] = round(cm[key]["predicted_us"] / cm[key]["measured_us"] - 1.0, 4)
        out["cost_model"] = cm
    hr = lines["hole_recompute"]
    out["prefill"] = {"workload": "hole_recompute: 16 seqs x (8192 cached, 25% evicted in holes of 2-32 blocks, "
                                  "recomputed) + 512-token turn, 32/8 heads, D=128",
                      "value": hr["prefill_tflops"], "unit": "TFLOP/s",
                      "roofline": {"bound": "tensor", "achieved": hr["prefill_tflops"],
                                   "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                   "frac": hr.get("tensor_frac"),
                                   "peak_source": f"bf16_tflops (burst, of {peak_src})",
                                   "traffic": hr.get("traffic")}}
    out["workloads"] = lines
    out["segmentation_overhead"] = over
    out["gather_then_attention"] = gathers
    out["eviction_policies"] = eviction_leg(dev, stream, steps, warm)
    out["prefill_chunking"] = chunking_leg(dev, stream, steps, warm)
    out["decode_shapes"] = decode_shapes_leg(dev, stream, peaks, steps, warm, rank)
    out["prefill_shapes"] = prefill_shapes_leg(dev, stream, peaks, steps, warm, rank)
    return out


# Hole recompute + new turn at other GQA ratios and head dims: (Hq, Hkv, D).
PREFILL_SHAPES = ((8, 8, 128), (24, 8, 128), (32, 8, 64))


def prefill_shapes_leg(dev, stream, peaks, steps, warm, rank):
    """Prefill tensor rate for odd G (query tiles are row pairs of one head)
    and D = 64."""
    import torch
    from kv_cache_segment_gb300 import workloads as W
    res = []
    for hq, hkv, d in PREFILL_SHAPES:
        wl = W.hole_recompute(seed=1003 + 1000 * rank, hq=hq, hkv=hkv, d=d)
        case = Case(wl, dev, plan_opts=_plan_opts())
        _, ms = time_case(case, steps, warm, stream, with_append=False)
        tf = case.flops() / (ms * 1e-3) / 1e12
        res.append({"hq": hq, "hkv": hkv, "head_dim": d, "G": hq // hkv, "attention_ms": round(ms, 4),
                    "prefill_tflops": round(tf, 1), "tensor_frac": round(tf / peaks["bf16_tflops"], 4),
                    "items": int(case.info["num_items"]), "model_predicted_us": _predict_us(case)})
        del case
        torch.cuda.empty_cache()
    return res


# Batched decode (the headline's length and segment draws) at other GQA
# ratios and head dimensions: (Hq, Hkv, D, sequences, pool tokens).  Each is
# sized so that the launch runs ~0.35-0.7 ms: a ~0.12 ms launch loses ~15-20 %
# to its fixed start and tail, which says nothing about the streaming rate.
DECODE_SHAPES = ((32, 32, 128, 32, 1 << 21), (64, 4, 128, 128, 1 << 23), (32, 8, 64, 128, 1 << 23),
                 (8, 8, 64, 128, 1 << 23))


def decode_shapes_leg(dev, stream, peaks, steps, warm, rank):
    """Decode HBM rate of the kernel across G = Hq/Hkv in {1, 16} and D = 64."""
    import torch
    from kv_cache_segment_gb300 import workloads as W
    res = []
    for hq, hkv, d, n, pool in DECODE_SHAPES:
        wl = W.batched_decode(seed=1002 + 1000 * rank, num_seqs=n, hq=hq, hkv=hkv, d=d, pool_tokens=pool)
        case = Case(wl, dev, plan_opts=_plan_opts())
        _, ms = time_case(case, steps, warm, stream, with_append=False)
        gbs = case.decode_bytes() / (ms * 1e-3) / 1e9
        res.append({"hq": hq, "hkv": hkv, "head_dim": d, "G": hq // hkv, "seqs": n, "attention_ms": round(ms, 4),
                    "decode_gbs": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                    "items": int(case.info["num_items"]), "model_predicted_us": _predict_us(case)})
        del case
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------- CPU legs --

def cpu_baseline(wl, target_s=15.0):
    """The float64 oracle, as it stands, on the host cores: a bounded sample
    of the same workload (the first sequences, all heads), repeated until
    about `target_s` seconds of CPU work; GB/s of the same algorithmic bytes."""
    import oracle
    from kv_cache_segment_gb300 import workloads as W
    threads = oracle.default_threads()
    n_seq = 1
    while True:
        sub = _subset(wl, n_seq)
        k, v, q = W.make_values(sub)
        t0 = time.perf_counter()
        oracle.dense_attention(sub.kv_indptr, k, v, sub.q_indptr, sub.q_pos, q, sub.num_q_heads,
                               sub.num_kv_heads, sub.scale, num_threads=threads)
        dt = time.perf_counter() - t0
        if dt >= target_s / 10 or n_seq >= wl.num_seqs:
            break
        n_seq = min(wl.num_seqs, n_seq * 2)
    kv = sum(min(int(sub.q_pos[sub.q_indptr[s + 1] - 1]) + 1, int(sub.seq_lens[s])) for s in range(sub.num_seqs))
    b = kv * sub.num_kv_heads * sub.head_dim * 4 + sub.num_q_rows * sub.num_q_heads * (sub.head_dim * 4 + 4)
    elapsed, reps = dt, 1
    while elapsed < target_s:
        t0 = time.perf_counter()
        oracle.dense_attention(sub.kv_indptr, k, v, sub.q_indptr, sub.q_pos, q, sub.num_q_heads,
                               sub.num_kv_heads, sub.scale, num_threads=threads)
        elapsed += time.perf_counter() - t0
        reps += 1
    used = min(threads, sub.num_q_rows * sub.num_q_heads)
    return {"value": round(b * reps / elapsed / 1e9, 4), "unit": "GB/s", "cores": used, "kind": "oracle",
            "sample": f"float64 oracle over the first {n_seq} of {wl.num_seqs} sequences (all heads), "
                      f"{reps} runs, {elapsed:.1f} s"}


def _subset(wl, n):
    import dataclasses
    return dataclasses.replace(wl, seq_lens=wl.seq_lens[:n].copy(), block_table=wl.block_table[:n].copy(),
                               q_ranges=wl.q_ranges[:n], runs_drawn=wl.runs_drawn[:n])


def reference_main(args):
    """Reference arm: the float64 oracle timed on the host cores, on the
    headline workload's configuration and metric (bounded sample per step)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    from kv_cache_segment_gb300 import workloads as W
    oracle.build_oracle()
    wl = W.config(2)
    per_step = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    vals = []
    for i in range(args.warmup + args.steps):
        r = cpu_baseline(wl, target_s=per_step)
        if i >= args.warmup:
            vals.append(r)
    value = float(np.mean([r["value"] for r in vals]))
    cores = vals[-1]["cores"]
    # a full step of the workload (its algorithmic K/V + q/out/lse bytes) at the oracle's rate
    kv = sum(int(wl.seq_lens[s]) for s in range(wl.num_seqs))
    step_bytes = kv * wl.num_kv_heads * wl.head_dim * 4 + wl.num_q_rows * wl.num_q_heads * (wl.head_dim * 4 + 4)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(step_bytes / (value * 1e9) * 1e3, 1), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "batched_decode: 32 seqs x 1 decode row, 32/8 heads, D=128, block 16, "
                                   "L~U{2048..16384}, 1-8 segments/seq in a 4M-token pool"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": vals[-1]["sample"]},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def profile_main(args):
    """A small case of one workload for ncu: pools of a few GB (the K/V read
    per launch still far above L2), two warm-up launches, then three timed
    ones of msa_attention (and msa_append_kv before each)."""
    import torch
    from kv_cache_segment_gb300 import msa
    from kv_cache_segment_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    msa.load()
    if args.profile == "decode":
        wl = W.batched_decode(seed=1002, pool_tokens=1 << 19)
    elif args.profile == "prefill":
        wl = W.config(3)
    elif args.profile == "mixed":
        wl = W.config(5)
    elif args.profile == "prefill64":  # the head-dim-64 prefill shape of prefill_shapes
        wl = W.hole_recompute(seed=1003, hq=32, hkv=8, d=64)
    else:
        wl = W.long_context(seed=1004, num_seqs=1)
    case = Case(wl, dev, plan_opts=_plan_opts())
    stream = torch.cuda.current_stream(dev)
    for _ in range(5):
        case.append(stream)
        case.attention(stream)
    torch.cuda.synchronize()
    rc, word = case.sess.check_device()
    print(json.dumps({"profile": args.profile, "workload": wl.name, "items": case.info["num_items"],
                      "decode_kv_bytes": case.info["decode_kv_bytes"], "prefill_flops": case.info["prefill_flops"],
                      "device_status": rc}))
    return 0 if rc == 0 else 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["msa", "reference"], default="msa")
    ap.add_argument("--quick", action="store_true", help="headline only (no e2e, extras or CPU baseline)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--profile", choices=["decode", "prefill", "mixed", "long", "prefill64"], default=None,
                    help="run a small case for an ncu capture and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        return profile_main(args)
    if args.impl == "reference":
        return reference_main(args)
    return gpu_main(args)


if __name__ == "__main__":
    sys.exit(main())
