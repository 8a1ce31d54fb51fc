"""Convenience wrapper over the C ABI for callers holding torch tensors.

`MsaSession` builds a plan from host arrays, allocates its device workspace
(a torch uint8 tensor), uploads it, and forwards attention calls.  It only
marshals arguments; all work runs in libmsa.
"""
from __future__ import annotations


from . import msa


def check_tensor(t, name, dtypes, shape, device=None):
    """Raise unless `t` is a contiguous tensor of one of `dtypes` with the
    given shape (None entries match any size) on `device` (when given).  The
    C ABI takes bare pointers, so this is the last place a wrong tensor can
    be caught before a kernel reads or writes past it."""
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype}, expected one of {[str(d) for d in dtypes]}")
    if t.dim() != len(shape) or any(w is not None and int(g) != w for g, w in zip(t.shape, shape)):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")


class MsaSession:
    def __init__(self, num_q_heads, num_kv_heads, head_dim, block_table, seq_lens, q_range_indptr, q_ranges,
                 device="cuda", num_sms=0, softmax_scale=None, stream=None, decode_split=0.0, prefill_split=0.0,
                 choose_with=None):
        import torch
        self.dims = msa.make_dims(num_q_heads, num_kv_heads, head_dim, 16, softmax_scale)
        if decode_split or prefill_split or choose_with is not None:
            self.plan = msa.msa_plan_create_ex(self.dims, block_table, seq_lens, q_range_indptr, q_ranges, num_sms,
                                               decode_split, prefill_split, choose_with)
        else:
            self.plan = msa.msa_plan_create(self.dims, block_table, seq_lens, q_range_indptr, q_ranges, num_sms)
        self.info = msa.msa_plan_get_info(self.plan)
        self.ws_bytes = msa.msa_plan_workspace_bytes(self.plan)
        self.workspace = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=device)
        self.stream = stream
        msa.msa_plan_upload(self.plan, self.workspace, self.ws_bytes, self._stream())

    @classmethod
    def from_workload(cls, wl, device="cuda", num_sms=0, stream=None, **plan_options):
        """plan_options: decode_split, prefill_split, choose_with (see msa_plan_create_ex)."""
        return cls(wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.block_table, wl.seq_lens, wl.q_range_indptr,
                   wl.q_ranges_flat, device=device, num_sms=num_sms, softmax_scale=wl.scale, stream=stream,
                   **plan_options)

    def _stream(self):
        import torch
        return self.stream if self.stream is not None else torch.cuda.current_stream()

    def attention(self, q, k_pool, v_pool, out=None, lse=None, out_fp32=False):
        """out (bf16, or fp32 with out_fp32 or an fp32 `out`) = attention of
        every query row of the plan; q bf16 [rows, Hq, D] in the plan's row
        order, pools bf16 [pool_tokens, Hkv, D], lse fp32 [rows, Hq] or None."""
        import torch
        hq, hkv, d = self.dims.num_q_heads, self.dims.num_kv_heads, self.dims.head_dim
        n_q = self.info["num_q_rows"]
        check_tensor(q, "q", (torch.bfloat16,), (n_q, hq, d))
        dev = q.device
        check_tensor(k_pool, "k_pool", (torch.bfloat16,), (None, hkv, d), dev)
        check_tensor(v_pool, "v_pool", (torch.bfloat16,), tuple(k_pool.shape), dev)
        if out is None:
            out = torch.empty((n_q, hq, d), dtype=torch.float32 if out_fp32 else torch.bfloat16, device=dev)
        check_tensor(out, "out", (torch.bfloat16, torch.float32), (n_q, hq, d), dev)
        if lse is not None:
            check_tensor(lse, "lse", (torch.float32,), (n_q, hq), dev)
        out_dtype = msa.MSA_OUT_FP32 if out.dtype == torch.float32 else msa.MSA_OUT_BF16
        msa.msa_attention(q, k_pool, v_pool, k_pool.shape[0], self.plan, out, out_dtype, lse, self._stream())
        return out

    def check_device(self):
        return msa.msa_plan_check_device(self.plan, self._stream())

    def close(self):
        if self.plan:
            msa.msa_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def append_kv(k_new, v_new, slot_mapping, k_pool, v_pool, dims, error_word=None, stream=None):
    """k_pool[slot[t]] = k_new[t], v_pool[slot[t]] = v_new[t] (slot -1 skips)."""
    import torch
    n, hkv, d = k_new.shape[0], dims.num_kv_heads, dims.head_dim
    check_tensor(k_new, "k_new", (torch.bfloat16,), (n, hkv, d))
    dev = k_new.device
    check_tensor(v_new, "v_new", (torch.bfloat16,), (n, hkv, d), dev)
    check_tensor(slot_mapping, "slot_mapping", (torch.int64,), (n,), dev)
    check_tensor(k_pool, "k_pool", (torch.bfloat16,), (None, hkv, d), dev)
    check_tensor(v_pool, "v_pool", (torch.bfloat16,), tuple(k_pool.shape), dev)
    if error_word is not None:
        check_tensor(error_word, "error_word", (torch.int32,), (None,), dev)
    msa.msa_append_kv(k_new, v_new, slot_mapping, k_new.shape[0], k_pool, v_pool, k_pool.shape[0], dims,
                      error_word, stream if stream is not None else torch.cuda.current_stream())
