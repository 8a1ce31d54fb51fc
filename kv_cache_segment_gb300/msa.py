"""ctypes binding of libmsa (include/msa.h), same names as the C ABI.

Argument marshalling only: every step of the path runs in the library's
CUDA kernels and C++ planner.  Pointers may be given as ints or as objects
with a ``data_ptr()`` method (torch tensors); streams as ints, torch streams
or None.  A failing call raises MsaError carrying the status code.  There is
no fallback: if libmsa.so is missing this module fails to import its
functions with an error saying how to build it.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmsa.so")

MSA_OK = 0
MSA_ERR_INVALID_ARG = -1
MSA_ERR_BAD_BLOCK_ID = -2
MSA_ERR_MISSING_BLOCK = -3
MSA_ERR_BAD_Q_RANGE = -4
MSA_ERR_WORKSPACE_TOO_SMALL = -5
MSA_ERR_UNSUPPORTED_DIMS = -6
MSA_ERR_CUDA = -7
MSA_ERR_DEVICE_CHECK = -8
MSA_ERR_NOT_UPLOADED = -9
MSA_OUT_BF16 = 0
MSA_OUT_FP32 = 1
MSA_EVICT_LINEAR = 0
MSA_EVICT_EXPECTED_COST = 1
MSA_EVICT_PREFIX_COST = 2  # OR-ed into either mode: the prefix reading of the recompute cost
MSA_DEVERR_TIMEOUT_PRODUCER = 1 << 0
MSA_DEVERR_TIMEOUT_MMA = 1 << 1
MSA_DEVERR_TIMEOUT_COMPUTE = 1 << 2
MSA_DEVERR_BAD_INDEX = 1 << 3
MSA_DEVERR_SLOT = 1 << 4
MSA_DEVERR_TMEM_ALLOC = 1 << 5


class MsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {msa_status_string(status)} ({status})")


class msa_dims(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float)]


class msa_plan_info(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_q_rows", ctypes.c_int32),
                ("num_runs", ctypes.c_int32), ("num_groups", ctypes.c_int32),
                ("num_items", ctypes.c_int32), ("num_decode_items", ctypes.c_int32),
                ("num_prefill_items", ctypes.c_int32), ("num_decode_rows", ctypes.c_int32),
                ("num_prefill_rows", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("decode_kv_bytes", ctypes.c_int64), ("decode_qo_bytes", ctypes.c_int64),
                ("prefill_flops", ctypes.c_double), ("max_pool_row", ctypes.c_int64),
                ("host_plan_us", ctypes.c_double), ("decode_split", ctypes.c_double),
                ("prefill_split", ctypes.c_double), ("counters_offset", ctypes.c_int64),
                ("counters_bytes", ctypes.c_int64)]


class msa_cost_params(ctypes.Structure):
    _fields_ = [("launch_us", ctypes.c_double), ("dec_item_us", ctypes.c_double),
                ("dec_gbs", ctypes.c_double), ("dec_cta_gbs", ctypes.c_double),
                ("pre_item_us", ctypes.c_double), ("pre_tile_us", ctypes.c_double),
                ("box_us", ctypes.c_double), ("dec_merge_us", ctypes.c_double),
                ("pre_merge_us", ctypes.c_double), ("pre_tile_dfrac", ctypes.c_double)]


class msa_cost_estimate(ctypes.Structure):
    _fields_ = [("time_us", ctypes.c_double), ("makespan_us", ctypes.c_double),
                ("fixed_us", ctypes.c_double), ("n_items", ctypes.c_int64),
                ("n_split_items", ctypes.c_int64), ("decode_tiles", ctypes.c_int64),
                ("prefill_tile_heads", ctypes.c_int64), ("extra_boxes", ctypes.c_int64),
                ("stream_bytes", ctypes.c_int64), ("decode_kv_bytes", ctypes.c_int64),
                ("prefill_flops", ctypes.c_double)]


COST_PARAM_NAMES = tuple(name for name, _ in msa_cost_params._fields_)


def _cost_params(d) -> msa_cost_params:
    """msa_cost_params from a dict of its field names.  A set without
    pre_tile_dfrac (one fitted with no head-dim term) prices a tile the same
    at every head dim, i.e. pre_tile_dfrac = 0."""
    return msa_cost_params(*[float(d.get(k, 0.0) if k == "pre_tile_dfrac" else d[k]) for k in COST_PARAM_NAMES])


class msa_pending_prefill(ctypes.Structure):
    _fields_ = [("seq", ctypes.c_int32), ("start", ctypes.c_int32), ("end", ctypes.c_int32)]


class msa_chunk_choice(ctypes.Structure):
    _fields_ = [("chunk", ctypes.c_int32), ("tokens", ctypes.c_int32), ("time_us", ctypes.c_double),
                ("us_per_token", ctypes.c_double), ("within_budget", ctypes.c_int32),
                ("n_candidates", ctypes.c_int32)]


class msa_plan_options(ctypes.Structure):
    _fields_ = [("num_sms", ctypes.c_int32), ("decode_split", ctypes.c_double),
                ("prefill_split", ctypes.c_double), ("choose_with", ctypes.POINTER(msa_cost_params))]

_lib = None


def load(path: str = LIB_PATH):
    """Load libmsa.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} not found: build it with `python -m kv_cache_segment_gb300.build`; "
                          "there is no fallback implementation")
    lib = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    sigs = {
        "msa_plan_create": ([ctypes.POINTER(msa_dims), i32, i32, vp, vp, vp, vp, i32, ctypes.POINTER(vp)], ctypes.c_int),
        "msa_plan_create_ex": ([ctypes.POINTER(msa_dims), i32, i32, vp, vp, vp, vp, ctypes.POINTER(msa_plan_options),
                                ctypes.POINTER(vp)], ctypes.c_int),
        "msa_plan_workspace_bytes": ([vp, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
        "msa_plan_upload": ([vp, vp, ctypes.c_size_t, vp], ctypes.c_int),
        "msa_plan_get_runs": ([vp, i32, vp, ctypes.POINTER(i32)], ctypes.c_int),
        "msa_plan_get_info": ([vp, ctypes.POINTER(msa_plan_info)], ctypes.c_int),
        "msa_plan_get_items": ([vp, vp, ctypes.POINTER(i32)], ctypes.c_int),
        "msa_plan_get_order": ([vp, vp, ctypes.POINTER(i32)], ctypes.c_int),
        "msa_plan_estimate": ([vp, ctypes.POINTER(msa_cost_params), ctypes.POINTER(msa_cost_estimate)],
                              ctypes.c_int),
        "msa_plan_destroy": ([vp], ctypes.c_int),
        "msa_choose_prefill_chunk": ([ctypes.POINTER(msa_dims), i32, i32, vp, vp, vp, vp, vp, i32,
                                      ctypes.POINTER(msa_plan_options), ctypes.POINTER(msa_cost_params),
                                      ctypes.c_double, i32, i32, ctypes.POINTER(msa_chunk_choice), vp, vp],
                                     ctypes.c_int),
        "msa_select_evictions": ([ctypes.POINTER(msa_dims), i32, vp, i32, ctypes.c_double, ctypes.c_double,
                                  ctypes.POINTER(msa_cost_params), i32, vp, vp], ctypes.c_int),
        "msa_append_kv": ([vp, vp, vp, i32, vp, vp, i64, ctypes.POINTER(msa_dims), vp, vp], ctypes.c_int),
        "msa_selftest_wait_timeout": ([ctypes.c_uint64, vp, vp], ctypes.c_int),
        "msa_gather_kv": ([vp, vp, i64, vp, i32, vp, vp, ctypes.POINTER(msa_dims), vp, vp], ctypes.c_int),
        "msa_attention": ([vp, vp, vp, i64, vp, vp, i32, vp, vp], ctypes.c_int),
        "msa_attention_no_alloc": ([vp, vp, vp, i64, vp, vp, i32, vp, vp], ctypes.c_int),
        "msa_plan_check_device": ([vp, vp, ctypes.POINTER(i32)], ctypes.c_int),
        "msa_no_alloc_check_device": ([vp, ctypes.POINTER(i32)], ctypes.c_int),
        "msa_no_alloc_inject_error": ([i32, vp], ctypes.c_int),
        "msa_status_string": ([ctypes.c_int], ctypes.c_char_p),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _p(x):
    """Pointer value of an int, None, numpy array or torch tensor."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot take a pointer of {type(x)}")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    raise TypeError(f"not a stream: {type(s)}")


def _check(rc: int, where: str):
    if rc != MSA_OK:
        raise MsaError(rc, where)


def make_dims(num_q_heads, num_kv_heads, head_dim, block_size=16, softmax_scale=None) -> msa_dims:
    if softmax_scale is None:
        softmax_scale = 1.0 / float(head_dim) ** 0.5
    return msa_dims(int(num_q_heads), int(num_kv_heads), int(head_dim), int(block_size), float(softmax_scale))


def msa_status_string(status: int) -> str:
    return load().msa_status_string(int(status)).decode()


def msa_plan_create(dims: msa_dims, block_table, seq_lens, q_range_indptr, q_ranges, num_sms: int = 0):
    """Host arrays in, opaque plan handle (int) out."""
    lib = load()
    table = np.ascontiguousarray(block_table, np.int32)
    if table.ndim != 2:
        table = table.reshape(len(seq_lens), -1)
    lens = np.ascontiguousarray(seq_lens, np.int32)
    indptr = np.ascontiguousarray(q_range_indptr, np.int32)
    ranges = np.ascontiguousarray(q_ranges, np.int32).reshape(-1, 2)
    plan = ctypes.c_void_p()
    rc = lib.msa_plan_create(ctypes.byref(dims), len(lens), table.shape[1], table.ctypes.data, lens.ctypes.data,
                             indptr.ctypes.data, ranges.ctypes.data if ranges.size else None, int(num_sms),
                             ctypes.byref(plan))
    _check(rc, "msa_plan_create")
    return plan.value


def msa_plan_create_ex(dims: msa_dims, block_table, seq_lens, q_range_indptr, q_ranges, num_sms: int = 0,
                       decode_split: float = 0.0, prefill_split: float = 0.0, choose_with=None):
    """msa_plan_create with explicit split factors, or (choose_with = a dict of
    msa_cost_params) factors chosen by the latency model."""
    lib = load()
    table = np.ascontiguousarray(block_table, np.int32)
    if table.ndim != 2:
        table = table.reshape(len(seq_lens), -1)
    lens = np.ascontiguousarray(seq_lens, np.int32)
    indptr = np.ascontiguousarray(q_range_indptr, np.int32)
    ranges = np.ascontiguousarray(q_ranges, np.int32).reshape(-1, 2)
    params = None
    if choose_with is not None:
        params = _cost_params(choose_with)
    opts = msa_plan_options(int(num_sms), float(decode_split), float(prefill_split),
                            ctypes.pointer(params) if params is not None else None)
    plan = ctypes.c_void_p()
    rc = lib.msa_plan_create_ex(ctypes.byref(dims), len(lens), table.shape[1], table.ctypes.data, lens.ctypes.data,
                                indptr.ctypes.data, ranges.ctypes.data if ranges.size else None, ctypes.byref(opts),
                                ctypes.byref(plan))
    _check(rc, "msa_plan_create_ex")
    return plan.value


def msa_choose_prefill_chunk(dims: msa_dims, block_table, seq_lens, q_range_indptr, q_ranges, pending, params,
                             budget_us: float = 0.0, granularity: int = 0, max_chunk: int = 0, num_sms: int = 0,
                             decode_split: float = 0.0, prefill_split: float = 0.0):
    """Chunk size for the pending prefills (list of (seq, start, end)) that
    minimises the predicted step time per prefill token within budget_us;
    returns (choice dict, candidates int32[n], predicted times float64[n]).
    params: dict of msa_cost_params names."""
    lib = load()
    table = np.ascontiguousarray(block_table, np.int32)
    if table.ndim != 2:
        table = table.reshape(len(seq_lens), -1)
    lens = np.ascontiguousarray(seq_lens, np.int32)
    indptr = np.ascontiguousarray(q_range_indptr, np.int32)
    ranges = np.ascontiguousarray(q_ranges, np.int32).reshape(-1, 2)
    pend = (msa_pending_prefill * max(1, len(pending)))(*[msa_pending_prefill(*map(int, p)) for p in pending])
    c = _cost_params(params)
    opts = msa_plan_options(int(num_sms), float(decode_split), float(prefill_split), None)
    choice = msa_chunk_choice()
    cand = np.zeros(64, np.int32)
    times = np.zeros(64, np.float64)
    _check(lib.msa_choose_prefill_chunk(ctypes.byref(dims), len(lens), table.shape[1], table.ctypes.data,
                                        lens.ctypes.data, indptr.ctypes.data,
                                        ranges.ctypes.data if ranges.size else None, pend, len(pending),
                                        ctypes.byref(opts), ctypes.byref(c), float(budget_us), int(granularity),
                                        int(max_chunk), ctypes.byref(choice), cand.ctypes.data, times.ctypes.data),
           "msa_choose_prefill_chunk")
    n = choice.n_candidates
    return {name: getattr(choice, name) for name, _ in msa_chunk_choice._fields_}, cand[:n], times[:n]


def msa_plan_workspace_bytes(plan) -> int:
    n = ctypes.c_size_t(0)
    _check(load().msa_plan_workspace_bytes(plan, ctypes.byref(n)), "msa_plan_workspace_bytes")
    return n.value


def msa_plan_upload(plan, workspace, nbytes: int, stream=None):
    _check(load().msa_plan_upload(plan, _p(workspace), int(nbytes), _stream(stream)), "msa_plan_upload")


def msa_plan_get_runs(plan, seq: int) -> np.ndarray:
    lib = load()
    n = ctypes.c_int32(0)
    _check(lib.msa_plan_get_runs(plan, int(seq), None, ctypes.byref(n)), "msa_plan_get_runs")
    out = np.zeros((max(n.value, 1), 3), np.int32)
    _check(lib.msa_plan_get_runs(plan, int(seq), out.ctypes.data, ctypes.byref(n)), "msa_plan_get_runs")
    return out[: n.value]


def msa_plan_get_info(plan) -> dict:
    info = msa_plan_info()
    _check(load().msa_plan_get_info(plan, ctypes.byref(info)), "msa_plan_get_info")
    return {name: getattr(info, name) for name, _ in msa_plan_info._fields_}


def msa_plan_get_items(plan) -> np.ndarray:
    lib = load()
    n = ctypes.c_int32(0)
    _check(lib.msa_plan_get_items(plan, None, ctypes.byref(n)), "msa_plan_get_items")
    out = np.zeros((max(n.value, 1), 9), np.int32)
    _check(lib.msa_plan_get_items(plan, out.ctypes.data, ctypes.byref(n)), "msa_plan_get_items")
    return out[: n.value]


def msa_plan_get_order(plan) -> np.ndarray:
    lib = load()
    n = ctypes.c_int32(0)
    _check(lib.msa_plan_get_order(plan, None, ctypes.byref(n)), "msa_plan_get_order")
    out = np.zeros(max(n.value, 1), np.int32)
    _check(lib.msa_plan_get_order(plan, out.ctypes.data, ctypes.byref(n)), "msa_plan_get_order")
    return out[: n.value]


def msa_plan_estimate(plan, params) -> dict:
    """Expected launch time and work features of a plan (see include/msa.h);
    `params` is a dict with the msa_cost_params field names."""
    c = _cost_params(params)
    e = msa_cost_estimate()
    _check(load().msa_plan_estimate(plan, ctypes.byref(c), ctypes.byref(e)), "msa_plan_estimate")
    return {name: getattr(e, name) for name, _ in msa_cost_estimate._fields_}


def msa_select_evictions(dims: msa_dims, seq_len: int, hit_prob, alpha: float, beta: float, params, n_evict: int,
                         mode: int = 0):
    """(evicted block indices ascending, per-block recompute cost in us) for
    one sequence; params: dict of msa_cost_params names (see include/msa.h)."""
    lib = load()
    hp = np.ascontiguousarray(hit_prob, np.float32)
    nb = -(-int(seq_len) // 16)
    ev = np.zeros(max(int(n_evict), 1), np.int32)
    cost = np.zeros(max(nb, 1), np.float64)
    c = _cost_params(params)
    _check(lib.msa_select_evictions(ctypes.byref(dims), int(seq_len), hp.ctypes.data if hp.size else None,
                                    int(mode), float(alpha), float(beta), ctypes.byref(c), int(n_evict),
                                    ev.ctypes.data, cost.ctypes.data), "msa_select_evictions")
    return ev[: int(n_evict)], cost[:nb]


def msa_plan_destroy(plan):
    if plan:
        load().msa_plan_destroy(plan)


def msa_append_kv(k_new, v_new, slot_mapping, n: int, k_pool, v_pool, pool_tokens: int, dims: msa_dims,
                  error_word=None, stream=None):
    _check(load().msa_append_kv(_p(k_new), _p(v_new), _p(slot_mapping), int(n), _p(k_pool), _p(v_pool),
                                int(pool_tokens), ctypes.byref(dims), _p(error_word), _stream(stream)),
           "msa_append_kv")


def msa_selftest_wait_timeout(limit_ns: int, device_words, stream=None):
    _check(load().msa_selftest_wait_timeout(int(limit_ns), _p(device_words), _stream(stream)),
           "msa_selftest_wait_timeout")


def msa_gather_kv(k_pool, v_pool, pool_tokens: int, slot_mapping, n: int, k_out, v_out, dims: msa_dims,
                  error_word=None, stream=None):
    _check(load().msa_gather_kv(_p(k_pool), _p(v_pool), int(pool_tokens), _p(slot_mapping), int(n), _p(k_out),
                                _p(v_out), ctypes.byref(dims), _p(error_word), _stream(stream)), "msa_gather_kv")


def msa_attention(q, k_pool, v_pool, pool_tokens: int, plan, out, out_dtype: int = MSA_OUT_BF16, lse=None,
                  stream=None):
    _check(load().msa_attention(_p(q), _p(k_pool), _p(v_pool), int(pool_tokens), plan, _p(out), int(out_dtype),
                                _p(lse), _stream(stream)), "msa_attention")


def msa_attention_no_alloc(q, k_pool, v_pool, pool_tokens: int, plan, out, out_dtype: int = MSA_OUT_BF16,
                           lse=None, stream=None):
    """msa_attention without a caller workspace (library-owned 32 MiB device
    array; see include/msa.h for who needs it and its limits)."""
    _check(load().msa_attention_no_alloc(_p(q), _p(k_pool), _p(v_pool), int(pool_tokens), plan, _p(out),
                                         int(out_dtype), _p(lse), _stream(stream)), "msa_attention_no_alloc")


def msa_plan_check_device(plan, stream=None):
    """(status, raw error word): synchronises the stream."""
    word = ctypes.c_int32(0)
    rc = load().msa_plan_check_device(plan, _stream(stream), ctypes.byref(word))
    return rc, word.value


def msa_no_alloc_check_device(stream=None):
    """(status, raw error word) of the last msa_attention_no_alloc call on the
    current device; synchronises the stream and clears a nonzero word."""
    word = ctypes.c_int32(0)
    rc = load().msa_no_alloc_check_device(_stream(stream), ctypes.byref(word))
    return rc, word.value


def msa_no_alloc_inject_error(bits: int, stream=None):
    """Test hook: OR `bits` into the no-alloc error word on `stream`."""
    _check(load().msa_no_alloc_inject_error(int(bits), _stream(stream)), "msa_no_alloc_inject_error")
