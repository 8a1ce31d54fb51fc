"""Fit the attention-latency model (msa_plan_estimate, include/msa.h) to
kernel times measured on this GPU, and check it on workloads it was not fitted
on.

AsymCache weighs recompute cost against hit rate with the attention kernel's
expected latency (MSA paper abstract; AsymCache explainer, "核心方法 2/3");
this script gives that model its constants for this kernel and GPU.

    python -m kv_cache_segment_gb300.costfit --out cost_params_gb300.json \
        --table ../profiles/latency_model_fit.md

Training and validation workloads are synthetic, drawn with the same
generators as the bench (decode batches of several sizes, lengths and
segment counts; hole recompute, also at odd GQA ratios; long-context
chunks; mixed batches; head dim 64 besides 128; and the bench's four
workloads at full size) at
different seeds and sizes for the two sets, each planned with three
different split factors (msa_plan_create_ex).  Each plan is timed as the median of
`--reps` launches of msa_attention alone (CUDA events on the launching
stream, after warm-up launches).  The ten parameters are fitted by
bounded least squares on log(predicted / measured).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import sys
import time

import numpy as np

from . import msa
from . import workloads as W

_HERE = os.path.dirname(os.path.abspath(__file__))
DEFAULT_PATH = os.path.join(_HERE, "cost_params_gb300.json")


def _decode(seed, n, lr, seg, name, hq=32, hkv=8):
    """A decode batch in a pool of twice its largest possible size (the
    generator scatters the segments over the whole pool)."""
    pool = -(-2 * n * lr[1] // 16) * 16
    return name, W.batched_decode(seed=seed, num_seqs=n, len_range=lr, max_seg=seg, pool_tokens=pool, hq=hq, hkv=hkv)


def training_set():
    s = []
    for i, (n, lr, seg) in enumerate([(8, (512, 4096), 1), (32, (2048, 16384), 8), (96, (2048, 8192), 4),
                                      (16, (16384, 32768), 64), (64, (256, 2048), 16), (128, (4096, 8192), 2)]):
        s.append(_decode(2000 + i, n, lr, seg, f"decode{i}"))
    for i, (n, G) in enumerate([(24, 8), (48, 2)]):
        s.append(_decode(2010 + i, n, (2048, 16384), 8, f"decode_g{G}", hq=8 * G))
    for i, (n, cb, ev) in enumerate([(2, 128, 32), (8, 256, 64), (16, 512, 128), (4, 512, 256)]):
        s.append((f"holes{i}", W.hole_recompute(seed=2020 + i, num_seqs=n, cached_blocks=cb, evict_blocks=ev)))
    for i, (length, runs, chunk) in enumerate([(16384, 1, 512), (65536, 64, 2048), (32768, 16, 1024)]):
        s.append((f"long{i}", W.long_context(seed=2030 + i, num_seqs=1, length=length, n_runs=runs, chunk=chunk)))
    # odd Hq/Hkv: prefill items are two row tiles of one head
    s.append(("holes_g1", W.hole_recompute(seed=2026, num_seqs=8, cached_blocks=256, evict_blocks=64, hq=8, hkv=8)))
    # head dim 64: the share of a prefill tile's time that scales with D
    s.append(("holes_d64", W.hole_recompute(seed=2027, num_seqs=8, cached_blocks=512, evict_blocks=128, d=64)))
    s.append(("long_d64", W.long_context(seed=2036, num_seqs=1, length=65536, n_runs=32, chunk=2048, d=64)))
    s.append(("decode_d64", W.batched_decode(seed=2012, num_seqs=64, len_range=(2048, 16384), max_seg=8,
                                             pool_tokens=1 << 21, d=64)))
    # launches the size of the bench's prefill workloads
    s.append(("holes_big", W.hole_recompute(seed=2025, num_seqs=16, cached_blocks=512, evict_blocks=128)))
    s.append(("long_big", W.long_context(seed=2035, num_seqs=2, length=98304, n_runs=48, chunk=2048)))
    for i, (nd, npf, chunk) in enumerate([(16, 1, 512), (64, 4, 2048), (128, 2, 1024)]):
        s.append((f"mixed{i}", W.mixed_batch(seed=2040 + i, num_decode=nd, num_prefill=npf, chunk=chunk)))
    # the bench's workloads as the bench draws them (the model plans them)
    for idx, name in ((2, "bench_decode"), (3, "bench_holes"), (4, "bench_long"), (5, "bench_mixed")):
        s.append((name, W.config(idx)))
    return s


def validation_set():
    s = []
    for i, (n, lr, seg) in enumerate([(20, (1024, 8192), 3), (48, (8192, 16384), 32), (200, (512, 4096), 8)]):
        s.append(_decode(3000 + i, n, lr, seg, f"v_decode{i}"))
    for i, (n, cb, ev) in enumerate([(4, 384, 96), (12, 512, 64)]):
        s.append((f"v_holes{i}", W.hole_recompute(seed=3010 + i, num_seqs=n, cached_blocks=cb, evict_blocks=ev)))
    s.append(("v_holes_g3", W.hole_recompute(seed=3012, num_seqs=6, cached_blocks=384, evict_blocks=96, hq=24, hkv=8)))
    s.append(("v_holes_d64", W.hole_recompute(seed=3013, num_seqs=12, cached_blocks=384, evict_blocks=96, d=64)))
    s.append(("v_mixed_d64", W.mixed_batch(seed=3032, num_decode=48, num_prefill=2, chunk=1024, d=64)))
    s.append(("v_long", W.long_context(seed=3020, num_seqs=2, length=49152, n_runs=32, chunk=1536)))
    for i, (nd, npf, chunk) in enumerate([(32, 2, 1024), (96, 3, 2048)]):
        s.append((f"v_mixed{i}", W.mixed_batch(seed=3030 + i, num_decode=nd, num_prefill=npf, chunk=chunk)))
    return s


# Each workload is measured under these (decode_split, prefill_split) plans:
# the same work cut into more or fewer items, so that the per-item and merge
# constants are told apart from the per-tile ones.
SPLITS = ((3.0, 4.0), (1.0, 1.0), (6.0, 8.0))


def measure(wl, dev, reps=15, warmup=3, splits=SPLITS):
    """[(median msa_attention time in us, session)] for each split plan.  The
    launches run back to back, as in a serving loop or the bench, each
    bracketed by its own CUDA events, so a launch's time starts when the
    previous one ends and excludes the host's launch latency."""
    import torch
    from .runner import MsaSession
    k, v, q = W.make_values(wl, device=dev)
    kp, vp = W.make_pool(wl, k, v, fill=0.0)
    del k, v
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)
    res = []
    for ds, ps in splits:
        sess = MsaSession.from_workload(wl, device=dev, decode_split=ds, prefill_split=ps)
        for _ in range(warmup):
            sess.attention(q, kp, vp, out=out)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in ev:
            a.record(stream)
            sess.attention(q, kp, vp, out=out)
            b.record(stream)
        torch.cuda.synchronize()
        times = [a.elapsed_time(b) * 1e3 for a, b in ev]
        rc, word = sess.check_device()
        if rc != 0:
            raise RuntimeError(f"device error word {word:#x}")
        res.append((float(np.median(times)), sess))
    return res


def predict(plan, params):
    return msa.msa_plan_estimate(plan, params)["time_us"]


def fit(records, x0=None):
    """records: [(plan, measured_us)] -> params dict (least squares on logs)."""
    from scipy.optimize import least_squares
    names = list(msa.COST_PARAM_NAMES)
    x0 = np.asarray(x0 if x0 is not None else [5.0, 2.0, 6400.0, 80.0, 5.0, 1.0, 0.02, 5.0, 20.0, 0.5], float)
    start = dict(zip(names, x0))
    # pre_tile_dfrac only matters for prefill at a head dim other than 128;
    # with no such record nothing determines it, and it stays 0 (the same
    # tile time at every head dim)
    fixed = {}
    if all(predict(pl, dict(start, pre_tile_dfrac=0.0)) == predict(pl, dict(start, pre_tile_dfrac=1.0))
           for pl, _ in records):
        fixed["pre_tile_dfrac"] = 0.0
    free = [k for k in names if k not in fixed]
    # every constant is >= 0; pre_tile_dfrac is a share, <= 1
    upper = np.array([1.0 if k == "pre_tile_dfrac" else np.inf for k in free])

    def resid(x):
        p = dict(zip(free, x), **fixed)
        return np.array([math.log(max(predict(pl, p), 1e-3) / t) for pl, t in records])

    r = least_squares(resid, np.array([start[k] for k in free]), bounds=(np.zeros(len(free)), upper), x_scale="jac")
    got = dict(zip(free, (float(v) for v in r.x)), **fixed)
    return {k: got[k] for k in names}


def errors(records, params):
    e = [predict(pl, params) / t - 1.0 for pl, t in records]
    return {"mean_abs_rel_err": float(np.mean(np.abs(e))), "max_abs_rel_err": float(np.max(np.abs(e)))}


def write_table(path, doc, rows):
    """The per-plan measurements and predictions behind a fit, as text."""
    with open(path, "w") as f:
        f.write("# Latency model fit: measured msa_attention launches and predictions\n\n")
        f.write(f"Device {doc['device']} ({doc['sm_count']} SMs); command `{doc['command']}`.\n")
        f.write("Each row: the median of the launches of one plan (split factors decode/prefill), CUDA events.\n\n")
        f.write("Parameters: " + ", ".join(f"{k} {v:g}" for k, v in doc["params"].items()) + "\n\n")
        for which in ("train", "validation"):
            e = doc["fit"][which]
            f.write(f"## {which}: mean |error| {100 * e['mean_abs_rel_err']:.1f} %, "
                    f"max {100 * e['max_abs_rel_err']:.1f} %\n\n")
            f.write("| workload | split | items | measured us | predicted us | error |\n|---|---|---|---|---|---|\n")
            for r in rows[which]:
                err = r["predicted_us"] / r["measured_us"] - 1.0
                f.write(f"| {r['workload']} | {r['decode_split']:g}/{r['prefill_split']:g} | {r['items']} | "
                        f"{r['measured_us']:.1f} | {r['predicted_us']:.1f} | {100 * err:+.1f} % |\n")
            f.write("\n")


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=DEFAULT_PATH)
    ap.add_argument("--table", default=None, help="also write the per-plan records as a text table here")
    ap.add_argument("--reps", type=int, default=15)
    args = ap.parse_args(argv)
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    msa.load()
    t0 = time.time()
    rows = {"train": [], "validation": []}
    keep = {"train": [], "validation": []}
    for which, wls in (("train", training_set()), ("validation", validation_set())):
        for name, wl in wls:
            for us, sess in measure(wl, dev, reps=args.reps):
                info = sess.info
                rows[which].append({"workload": name, "decode_split": info["decode_split"],
                                    "prefill_split": info["prefill_split"], "measured_us": round(us, 2),
                                    "items": info["num_items"], "decode_kv_bytes": info["decode_kv_bytes"],
                                    "prefill_flops": info["prefill_flops"]})
                keep[which].append((sess, us))
                print(f"{which:10s} {name:12s} split {info['decode_split']:.1f}/{info['prefill_split']:.1f} "
                      f"{us:10.1f} us  items {info['num_items']}", file=sys.stderr)
            torch.cuda.empty_cache()
    train = [(s.plan, t) for s, t in keep["train"]]
    val = [(s.plan, t) for s, t in keep["validation"]]
    params = fit(train)
    for which, recs in (("train", train), ("validation", val)):
        for row, (pl, t) in zip(rows[which], recs):
            row["predicted_us"] = round(predict(pl, params), 2)
    doc = {
        "device": torch.cuda.get_device_name(dev),
        "sm_count": torch.cuda.get_device_properties(dev).multi_processor_count,
        "params": {k: round(v, 5) for k, v in params.items()},
        "fit": {"train": errors(train, params), "validation": errors(val, params)},
        "plans": {"train": len(train), "validation": len(val)},
        "seconds": round(time.time() - t0, 1),
        "command": "python -m kv_cache_segment_gb300.costfit --out <path> --table <path>",
    }
    with open(args.out, "w") as f:
        json.dump(doc, f, indent=1)
    if args.table:
        write_table(args.table, doc, rows)
    print(json.dumps({"params": doc["params"], "fit": doc["fit"]}))
    for s, _ in keep["train"] + keep["validation"]:
        s.close()
    return 0


def load_params(path: str = DEFAULT_PATH):
    """The fitted parameters (dict), or None when no fit has been stored."""
    if not os.path.exists(path):
        return None
    with open(path) as f:
        return json.load(f)["params"]


if __name__ == "__main__":
    sys.exit(main())
