"""msa_attention_no_alloc: attention for callers that may not allocate
device memory (a serving engine whose memory is carved up at start-up, a
plug-in without access to the host framework's allocator).  It keeps its
workspace in a library-owned device array; its results must match
msa_attention's, call after call.

Collected last on purpose: if it fails, a run stopped at the first failure
has already run every other test."""
import numpy as np
import pytest
import torch

from gpu_harness import compare, oracle_ref
from kv_cache_segment_gb300 import msa, workloads as W
from kv_cache_segment_gb300.runner import MsaSession

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    msa.load()


@pytest.mark.parametrize("idx", [5, 3])
def test_no_alloc_matches_msa_attention_twice(idx):
    wl = W.small_config(idx)
    k, v, q = W.make_values(wl)
    dev = torch.device("cuda")
    kp, vp = W.make_pool(wl, k.to(dev), v.to(dev))
    qd = q.to(dev)
    # many CTAs, so long groups are split and the merge counters are used
    sess = MsaSession.from_workload(wl, num_sms=600)
    lse_ref = torch.empty((wl.num_q_rows, wl.num_q_heads), dtype=torch.float32, device=dev)
    out_ref = sess.attention(qd, kp, vp, lse=lse_ref)
    assert sess.check_device()[0] == 0
    ro, rl = oracle_ref(wl, k, v, q)
    compare(out_ref, lse_ref, ro, rl, "msa_attention")
    stream = torch.cuda.current_stream()
    for call in range(2):
        out = torch.full_like(out_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        msa.msa_attention_no_alloc(qd, kp, vp, kp.shape[0], sess.plan, out, msa.MSA_OUT_BF16, lse, stream)
        torch.cuda.synchronize()
        o_ref = out_ref.float().cpu().numpy().astype(np.float64)
        l_ref = lse_ref.cpu().numpy().astype(np.float64)
        compare(out, lse, o_ref, l_ref, f"no_alloc call {call}")
        compare(out, lse, ro, rl, f"no_alloc call {call} vs oracle")
    sess.close()


def test_no_alloc_rejects_oversized_plan():
    # a plan whose workspace exceeds the 32 MiB array is refused, nothing launched
    wl = W.config(4)
    dims = msa.make_dims(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, 16, wl.scale)
    plan = msa.msa_plan_create(dims, wl.block_table, wl.seq_lens, wl.q_range_indptr, wl.q_ranges_flat, 5000)
    try:
        assert msa.msa_plan_workspace_bytes(plan) > (32 << 20)
        with pytest.raises(msa.MsaError) as e:
            msa.msa_attention_no_alloc(16, 16, 16, wl.pool_tokens, plan, 16)
        assert e.value.status == msa.MSA_ERR_WORKSPACE_TOO_SMALL
    finally:
        msa.msa_plan_destroy(plan)


def test_no_alloc_errors_are_visible_and_cleared():
    """msa_no_alloc_check_device reads the error word the no-alloc calls
    share: zero after clean calls; a word planted from the host (as a kernel
    that gave up would leave it) is reported once and cleared; a call after
    that is still exact."""
    wl = W.small_config(5)
    k, v, q = W.make_values(wl)
    dev = torch.device("cuda")
    kp, vp = W.make_pool(wl, k.to(dev), v.to(dev))
    qd = q.to(dev)
    sess = MsaSession.from_workload(wl, num_sms=600)
    stream = torch.cuda.current_stream()
    ro, rl = oracle_ref(wl, k, v, q)
    try:
        out = torch.empty((wl.num_q_rows, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((wl.num_q_rows, wl.num_q_heads), dtype=torch.float32, device=dev)
        msa.msa_attention_no_alloc(qd, kp, vp, kp.shape[0], sess.plan, out, msa.MSA_OUT_BF16, lse, stream)
        assert msa.msa_no_alloc_check_device(stream) == (msa.MSA_OK, 0)
        bits = msa.MSA_DEVERR_TIMEOUT_MMA | msa.MSA_DEVERR_BAD_INDEX
        msa.msa_no_alloc_inject_error(bits, stream)
        assert msa.msa_no_alloc_check_device(stream) == (msa.MSA_ERR_DEVICE_CHECK, bits)
        assert msa.msa_no_alloc_check_device(stream) == (msa.MSA_OK, 0)
        out.fill_(float("nan"))
        msa.msa_attention_no_alloc(qd, kp, vp, kp.shape[0], sess.plan, out, msa.MSA_OUT_BF16, lse, stream)
        assert msa.msa_no_alloc_check_device(stream) == (msa.MSA_OK, 0)
        compare(out, lse, ro, rl, "no_alloc after a reported error")
    finally:
        sess.close()
