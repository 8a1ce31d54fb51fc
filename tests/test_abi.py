"""The C-ABI library loads and exports every function include/msa.h declares
(no GPU needed: nothing here launches a kernel)."""
import ctypes
import os
import re

from kv_cache_segment_gb300 import msa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[\w\*]+\s+\*?(msa_\w+)\s*\(", txt, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert "msa_attention" in names and "msa_plan_create" in names and "msa_append_kv" in names
    lib = ctypes.CDLL(msa.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings():
    for code in range(0, -10, -1):
        s = msa.msa_status_string(code)
        assert s.startswith("MSA_")
    assert msa.msa_status_string(-1234) == "MSA_ERR_UNKNOWN"


def test_package_has_no_cpu_fallback():
    """The binding must not import the oracle (test infrastructure)."""
    import kv_cache_segment_gb300
    pkg = os.path.dirname(kv_cache_segment_gb300.__file__)
    for f in os.listdir(pkg):
        if f.endswith(".py"):
            src = open(os.path.join(pkg, f)).read()
            assert "import oracle" not in src and "from oracle" not in src, f


def test_argument_checks_return_before_any_device_work():
    """Checks the header documents that come back before a launch (fake,
    never dereferenced device addresses; nothing here needs a GPU)."""
    import ctypes as C
    lib = msa.load()
    dims = msa.make_dims(8, 2, 128)
    A, MIS = 0x10000, 0x10002  # 16-byte aligned / 2 bytes past a boundary
    ok, bad = msa.MSA_OK, msa.MSA_ERR_INVALID_ARG
    # msa_append_kv: n == 0 is a no-op even with NULL pointers; misaligned rows are refused
    assert lib.msa_append_kv(None, None, None, 0, None, None, 64, C.byref(dims), None, None) == ok
    for args in [(MIS, A, A, A, A), (A, MIS, A, A, A), (A, A, A, MIS, A), (A, A, A, A, MIS), (A, A, None, A, A)]:
        kn, vn, slot, kp, vp = args
        assert lib.msa_append_kv(kn, vn, slot, 4, kp, vp, 64, C.byref(dims), None, None) == bad, args
    assert lib.msa_append_kv(A, A, A, -1, A, A, 64, C.byref(dims), None, None) == bad
    odd = msa.make_dims(8, 2, 96)
    assert lib.msa_append_kv(A, A, A, 4, A, A, 64, C.byref(odd), None, None) == msa.MSA_ERR_UNSUPPORTED_DIMS
    # msa_gather_kv: the same rules
    assert lib.msa_gather_kv(None, None, 64, None, 0, None, None, C.byref(dims), None, None) == ok
    for args in [(MIS, A, A, A, A), (A, A, A, MIS, A), (A, A, A, A, MIS), (A, A, None, A, A)]:
        kp, vp, slot, ko, vo = args
        assert lib.msa_gather_kv(kp, vp, 64, slot, 4, ko, vo, C.byref(dims), None, None) == bad, args
    # msa_selftest_wait_timeout: limit in [1 ns, 10 s], words required
    assert lib.msa_selftest_wait_timeout(0, A, None) == bad
    assert lib.msa_selftest_wait_timeout(10_000_000_001, A, None) == bad
    assert lib.msa_selftest_wait_timeout(1000, None, None) == bad
    # msa_attention on a plan that was never uploaded, and without a plan
    assert lib.msa_attention(A, A, A, 64, None, A, 0, None, None) == bad
    import numpy as np
    plan = msa.msa_plan_create(dims, np.zeros((1, 1), np.int32), np.array([16], np.int32),
                               np.array([0, 1], np.int32), np.array([16, 17], np.int32), 4)
    try:
        assert lib.msa_attention(A, A, A, 64, plan, A, 0, None, None) == msa.MSA_ERR_NOT_UPLOADED
    finally:
        msa.msa_plan_destroy(plan)


def test_tensor_checks_of_the_python_wrapper():
    """runner.check_tensor, which MsaSession.attention and append_kv apply to
    every tensor before a pointer crosses the ABI."""
    import pytest
    import torch
    from kv_cache_segment_gb300.runner import check_tensor
    t = torch.zeros((5, 4, 64), dtype=torch.bfloat16)
    check_tensor(t, "t", (torch.bfloat16,), (5, 4, 64))
    check_tensor(t, "t", (torch.bfloat16,), (None, 4, 64))
    with pytest.raises(TypeError):
        check_tensor(t.float(), "t", (torch.bfloat16,), (5, 4, 64))
    with pytest.raises(ValueError):
        check_tensor(t, "t", (torch.bfloat16,), (5, 4, 128))
    with pytest.raises(ValueError):
        check_tensor(t, "t", (torch.bfloat16,), (5, 4))
    with pytest.raises(ValueError):
        check_tensor(t.transpose(0, 1), "t", (torch.bfloat16,), (4, 5, 64))
    with pytest.raises(ValueError):
        check_tensor(t, "t", (torch.bfloat16,), (5, 4, 64), torch.device("meta"))
