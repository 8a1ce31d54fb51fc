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


def compare(out, lse, ref_out, ref_lse, what="", extra=None):
    """Element-wise parity; `extra` (same shape as out, or None) is added to
    the out bound where a case's arithmetic allows more than the stated
    tolerance (see test_running_max_moves)."""
    out = out.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    assert out.shape == ref_out.shape and lse.shape == ref_lse.shape
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), f"{what}: lse finiteness differs"
    assert np.all(np.isneginf(lse[~fin])), what
    err = np.abs(out - ref_out)
    bound = OUT_ABS + OUT_REL * np.abs(ref_out)
    if extra is not None:
        bound = bound + extra
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
