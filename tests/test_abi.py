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
