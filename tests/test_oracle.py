"""The float64 oracle against facts that do not come from it (CPU only)."""
import pytest

import oracle_pins as P


@pytest.mark.parametrize("pin", P.ATTENTION_PINS, ids=lambda f: f.__name__)
def test_attention_pin(pin):
    pin()


def test_segment_splitter_pin():
    P.pin_segment_splitter()


def test_scatter_pin():
    P.pin_scatter()


def test_tiny_decode_layout_golden():
    import json
    import os
    import oracle
    from kv_cache_segment_gb300 import workloads as W
    with open(os.path.join(P.GOLDEN, "tiny_decode_layout.json")) as f:
        g = json.load(f)
    wl = W.config(1)
    runs = oracle.segment_runs(wl.block_table[0], g["seq_len"] // g["block_size"])
    assert [[int(r[0]), int(r[2])] for r in runs] == g["segments_logical"]
    # the three segments sit at distinct, non-adjacent pool offsets
    starts = sorted(int(r[1]) for r in runs)
    sizes = {int(r[1]): int(r[2]) for r in runs}
    for a, b in zip(starts, starts[1:]):
        assert b > a + sizes[a]
