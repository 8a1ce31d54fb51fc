"""The plain latency-model and eviction oracles against hand-worked closed
forms (model_pins.py), and copies of them with planted mistakes against the
same pins: every planted mistake must be caught (CPU only)."""
import importlib.util
import os
import shutil
import sys
import tempfile

import pytest

import model_pins as P
import oracle
import oracle.costmodel as OC
import oracle.eviction as OE

ORACLE_DIR = os.path.dirname(oracle.__file__)


@pytest.mark.parametrize("pin", P.COST_PINS, ids=lambda f: f.__name__)
def test_cost_oracle_pin(pin):
    pin(OC)


@pytest.mark.parametrize("pin", P.EVICTION_PINS, ids=lambda f: f.__name__)
def test_eviction_oracle_pin(pin):
    pin(OE)


# (module, name, text in the module, replacement)
MUTATIONS = [
    ("costmodel", "prefill_qtiles_dropped", "tile_us(params, head_dim) * tiles * qtiles",
     "tile_us(params, head_dim) * tiles"),
    ("costmodel", "tile_head_dim_ratio_inverted", "dfrac * head_dim / 128.0", "dfrac * 128.0 / head_dim"),
    ("costmodel", "tile_fixed_share_dropped", "((1.0 - dfrac) + dfrac * head_dim / 128.0)",
     "(dfrac * head_dim / 128.0)"),
    ("costmodel", "tile_shares_swapped", "((1.0 - dfrac) + dfrac * head_dim / 128.0)",
     "(dfrac + (1.0 - dfrac) * head_dim / 128.0)"),
    ("costmodel", "tile_head_dim_ignored", "tile_us(params, head_dim) * tiles * qtiles",
     'params["pre_tile_us"] * tiles * qtiles'),
    ("costmodel", "qtiles_ignore_rows", "qtiles = -(-nrows // TILE) * heads", "qtiles = heads"),
    ("costmodel", "stream_k_only", "tile_bytes = 2.0 * TILE * head_dim * 2.0", "tile_bytes = TILE * head_dim * 2.0"),
    ("costmodel", "bandwidth_not_shared", 'params["dec_gbs"] / n_stream', 'params["dec_gbs"]'),
    ("costmodel", "merge_for_every_item", "(merge if split else 0.0)", "merge"),
    ("costmodel", "merge_constants_swapped", 'params["dec_merge_us"] if kind == 0 else params["pre_merge_us"]',
     'params["pre_merge_us"] if kind == 0 else params["dec_merge_us"]'),
    ("costmodel", "one_box_per_piece", "boxes += b // 4 + (b % 4) // 2 + b % 2", "boxes += 1"),
    ("costmodel", "one_box_per_block", "boxes += b // 4 + (b % 4) // 2 + b % 2", "boxes += b"),
    ("costmodel", "queue_taken_last_first", "                    j = queue.pop(0)",
     "                    j = queue.pop()"),
    ("costmodel", "launch_left_out", 'out["time_us"] = params["launch_us"] + t', 'out["time_us"] = t'),
    ("costmodel", "recompute_row_misses_itself", "sum(min(p + 1, seq_len) for p in range(start, end))",
     "sum(min(p, seq_len) for p in range(start, end))"),
    ("costmodel", "chunk_budget_ignored", "if budget_us <= 0 or t <= budget_us]", "]"),
    ("costmodel", "chunk_total_time_not_per_token", "ok = [(t / n, -c, c)", "ok = [(t, -c, c)"),
    ("costmodel", "chunk_ties_to_the_smaller", "ok = [(t / n, -c, c)", "ok = [(t / n, c, c)"),
    ("costmodel", "chunk_cap_not_a_candidate", "    if not out or out[-1] != cap:\n        out.append(cap)\n",
     "    if not out:\n        out.append(cap)\n"),
    ("costmodel", "chunk_thinning_off_by_one", "step = max(1, -(-n_mult // 63))", "step = max(1, n_mult // 63)"),
    ("costmodel", "chunk_rows_not_capped_by_remainder", "n = min(c, b - a)", "n = c"),
    ("eviction", "cost_row_misses_itself", "keys += min(p + 1, seq_len)", "keys += min(p, seq_len)"),
    ("eviction", "cost_on_the_evict_side", "(beta * c / cmax if cmax > 0 else 0.0)",
     "(-beta * c / cmax if cmax > 0 else 0.0)"),
    ("eviction", "tile_area_wrong", "keys / (128 * 128)", "keys / 128"),
    ("eviction", "ties_to_higher_block", "key=lambda x: (x[0], x[1])", "key=lambda x: (x[0], -x[1])"),
    ("eviction", "expected_cost_added", "s = float(hit_prob[b]) * c", "s = float(hit_prob[b]) + c"),
    ("eviction", "keeps_the_lowest", "scored[:n_evict]", "scored[len(scored) - n_evict:]"),
    ("eviction", "prefix_sums_the_wrong_side", "sum(hole[b:])", "sum(hole[:b + 1])"),
    ("eviction", "prefix_leaves_the_block_out", "sum(hole[b:])", "sum(hole[b + 1:])"),
    ("eviction", "prefix_reading_ignored", "    if prefix:\n", "    if False:\n"),
]


def _load_mutant(tmp, module, name, old, new):
    pkg = os.path.join(tmp, f"mut_{name}")
    os.makedirs(pkg)
    open(os.path.join(pkg, "__init__.py"), "w").close()
    shutil.copy(os.path.join(ORACLE_DIR, "segments.py"), pkg)
    src = open(os.path.join(ORACLE_DIR, f"{module}.py")).read()
    assert src.count(old) == 1, f"mutation anchor missing or ambiguous: {name}"
    with open(os.path.join(pkg, f"{module}.py"), "w") as f:
        f.write(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"mut_{name}", os.path.join(pkg, "__init__.py"),
                                                  submodule_search_locations=[pkg])
    mod = importlib.util.module_from_spec(spec)
    sys.modules[spec.name] = mod
    spec.loader.exec_module(mod)
    return importlib.import_module(f"mut_{name}.{module}")


@pytest.mark.parametrize("module,name,old,new", MUTATIONS, ids=[m[1] for m in MUTATIONS])
def test_pins_catch_planted_model_mistake(module, name, old, new):
    pins = P.COST_PINS if module == "costmodel" else P.EVICTION_PINS
    with tempfile.TemporaryDirectory() as tmp:
        mut = _load_mutant(tmp, module, name, old, new)
        caught = []
        for pin in pins:
            try:
                pin(mut)
            except (AssertionError, ZeroDivisionError, ValueError):
                caught.append(pin.__name__)
        sys.modules.pop(f"mut_{name}", None)
        sys.modules.pop(f"mut_{name}.{module}", None)
        sys.modules.pop(f"mut_{name}.segments", None)
        assert caught, f"no pin caught the planted mistake {name}"
