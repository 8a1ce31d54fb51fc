"""Shared helpers of the GPU parity tests: run a workload through the C ABI
and compare with the float64 oracle element by element."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from kv_cache_segment_gb300 import workloads as W
from kv_cache_segment_gb300.runner import MsaSession

OUT_ABS = 2e-3   # |out - ref| <= OUT_ABS + OUT_REL * |ref|  (per element)
OUT_REL = 1e-2
LSE_ABS = 1e-4


def compare(out, lse, ref_out, ref_lse, what=""):
    """Element-wise parity at the stated tolerance: every out element within
    OUT_ABS + OUT_REL * |ref|, every finite lse within LSE_ABS."""
    out = out.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    assert out.shape == ref_out.shape and lse.shape == ref_lse.shape
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: lse finiteness differs"
    assert np.all(np.isneginf(lse[~fin])), what
    err = np.abs(out - ref_out)
    bound = OUT_ABS + OUT_REL * np.abs(ref_out)
    bad = ~(err <= bound)
    assert not bad.any(), (f"{what}: {bad.sum()} out elements beyond tolerance; max abs err "
                           f"{np.nanmax(err):.3e}; worst at {np.unravel_index(np.argmax(err - bound), err.shape)}")
    lerr = np.abs(lse[fin] - ref_lse[fin]) if fin.any() else np.zeros(1)
    assert lerr.max() <= LSE_ABS, f"{what}: lse max abs err {lerr.max():.3e}"
    big = np.abs(ref_out) >= 0.2
    rel = float((err[big] / np.abs(ref_out[big])).max()) if big.any() else 0.0
    return {"out_max_abs": float(err.max()), "out_max_rel": rel, "lse_max_abs": float(lerr.max())}


def run_gpu(wl, k_log, v_log, q, out_fp32=False, num_sms=0, fill=float("nan"), **plan_opts):
    """Pools from the logical K/V (other rows = `fill`), then plan+attention;
    plan_opts go to msa_plan_create_ex (decode_split, prefill_split,
    choose_with)."""
    dev = torch.device("cuda")
    kl, vl, qd = k_log.to(dev), v_log.to(dev), q.to(dev)
    kp, vp = W.make_pool(wl, kl, vl, fill=fill)
    sess = MsaSession.from_workload(wl, num_sms=num_sms, **plan_opts)
    lse = torch.empty((wl.num_q_rows, wl.num_q_heads), dtype=torch.float32, device=dev)
    out = sess.attention(qd, kp, vp, lse=lse, out_fp32=out_fp32)
    rc, word = sess.check_device()
    assert rc == 0, f"device error word {word:#x}"
    torch.cuda.synchronize()
    info = sess.info
    sess.close()
    return out, lse, info


def oracle_ref(wl, k_log, v_log, q, rows=None):
    return oracle.dense_attention(wl.kv_indptr, k_log, v_log, wl.q_indptr, wl.q_pos, q, wl.num_q_heads,
                                  wl.num_kv_heads, wl.scale, rows=rows)


def random_workload(seed):
    """A small seeded workload with its shape drawn too: D in {64, 128},
    Hkv in {1, 2, 4}, G = Hq/Hkv in {1, 2, 3, 4, 5, 8, 16} (at most 64 query
    heads), 1-5 sequences of 0-1500 cached tokens in 1-8 segments, 1-3
    disjoint query ranges per sequence (decode rows at p = L included; about
    a third of the sequences decode-only, 1 to 16/G trailing rows), and
    a plan option set (default, fine split, coarse).  N(0, 1) values as
    everywhere else."""
    rng = np.random.default_rng(10_000 + seed)
    d = int(rng.choice([64, 128]))
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([G for G in (1, 2, 3, 4, 5, 8, 16) if hkv * G <= 64]))
    n = int(rng.integers(1, 6))
    lens, runs, ranges = [], [], []
    for _ in range(n):
        L = int(rng.integers(0, 1501)) if rng.random() > 0.1 else 0
        nb = -(-L // 16)
        lens.append(L)
        runs.append(W._cut_sizes(rng, nb, int(rng.integers(1, 9))) if nb else [])
        # 1-3 sorted disjoint ranges inside [0, L + 1); the last often ends at L + 1 (decode)
        k = int(rng.integers(1, 4))
        cuts = np.sort(rng.choice(np.arange(0, L + 2), size=min(2 * k, L + 2), replace=False))
        rs = [(int(a), int(b)) for a, b in zip(cuts[0::2], cuts[1::2]) if b > a]
        rs = [(a, min(b, a + 300)) for a, b in rs]
        if rng.random() < 0.6 and (not rs or rs[-1][1] <= L):
            rs.append((L, L + 1))
        if rng.random() < 0.35:  # decode-only: the last 1 .. 16/G rows (the GQA-packed path)
            t = int(rng.integers(1, 16 // g + 1))
            rs = [(max(0, L + 1 - t), L + 1)]
        ranges.append(rs or [(L, L + 1)])
    opts = [dict(), dict(decode_split=12.0, prefill_split=16.0), dict(decode_split=1.0, prefill_split=1.0)][seed % 3]
    wl = W.custom(lens, runs, ranges, hq=hkv * g, hkv=hkv, d=d, seed=20_000 + seed)
    return wl, opts
