"""Plant plausible mistakes in copies of the oracle (on the CPU) and check
that the pins catch every one of them."""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
import oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement)
MUTATIONS = [
    ("causal_excludes_self", "int64_t n_vis = p + 1 < len ? p + 1 : len;",
     "int64_t n_vis = p < len ? p : len;"),
    ("gqa_head_modulo", "const int32_t g = h / group;\n            double* o",
     "const int32_t g = h % group;\n            double* o"),
    ("dropped_scale", "t[j] = jb->scale * acc;", "t[j] = acc;"),
    ("unnormalised_weights", "const double w = exp(t[j] - l);", "const double w = exp(t[j] - m);"),
    ("value_reads_keys", "const uint16_t* vj = jb->v + ((kv0 + j)", "const uint16_t* vj = jb->k + ((kv0 + j)"),
    ("lse_base2", "const double l = m + log(sum);\n            jb->lse", "const double l = m + log2(sum);\n            jb->lse"),
    ("merge_weight_unnormalised", "const double w = exp(lse_r[k] - LSE);", "const double w = exp(lse_r[k] - mx);"),
    ("segment_sees_future", "if (log1 > p + 1) log1 = p + 1;", "if (log1 > p + 2) log1 = p + 2;"),
    ("segment_ignores_physical_jump", "table[e] == table[e - 1] + 1", "table[e] >= table[e - 1]"),
    ("segment_wrong_pool_row", "((phys0 + (j - log0)) * hkv + g) * (int64_t)d;\n                    double acc",
     "((phys0 + (j - log0) + 1) * hkv + g) * (int64_t)d;\n                    double acc"),
]


def _build_variant(tmp, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor missing: {name}"
    src = src.replace(old, new, 1)
    path = os.path.join(tmp, f"{name}.c")
    with open(path, "w") as f:
        f.write(src)
    lib = os.path.join(tmp, f"lib_{name}.so")
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-D_GNU_SOURCE", "-shared", "-fPIC", "-pthread",
                           path, "-o", lib, "-lm"])
    return oracle.load_variant(lib)


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(name, old, new):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    with tempfile.TemporaryDirectory() as tmp:
        lib = _build_variant(tmp, name, old, new)
        caught = []
        for pin in P.ATTENTION_PINS:
            try:
                pin(lib=lib)
            except AssertionError:
                caught.append(pin.__name__)
            except (RuntimeError, ValueError):
                caught.append(pin.__name__ + "(error)")
        assert caught, f"no pin caught the planted mistake {name}"
