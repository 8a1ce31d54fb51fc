"""include/msa.h is a C header and libmsa.so is callable from plain C: a C11
program (tests/c_abi/plan_from_c.c) built with gcc against them runs the
host-only calls (CPU only)."""
import os
import shutil
import subprocess

import pytest

from kv_cache_segment_gb300 import msa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_plain_c_caller(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    exe = str(tmp_path / "plan_from_c")
    libdir = os.path.dirname(msa.LIB_PATH)
    subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                           os.path.join(ROOT, "tests", "c_abi", "plan_from_c.c"), "-o", exe, "-L", libdir, "-lmsa",
                           "-Wl,-rpath," + libdir])
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    lines = out.stdout.splitlines()
    got = lines[0].split()
    vals = dict(zip(got[0::2], got[1::2]))
    # 11 prefill rows + 1 decode row; seq 0 = runs (block 0, phys 10, 2 blocks) and (block 2, phys 17, 1 block)
    assert vals["rows"] == "12" and vals["runs"] == "2"
    assert got[got.index("run0") + 1:got.index("run0") + 4] == ["0", "10", "2"]
    assert got[got.index("run1") + 1:got.index("run1") + 4] == ["2", "17", "1"]
    assert int(vals["items"]) >= 2 and vals["ws_ok"] == "1" and vals["est_items"] == vals["items"]
    assert vals["evict"] == "1"  # alpha only: the block least likely to be hit
    assert vals["cost_rising"] == "1" and vals["not_uploaded"] == "MSA_ERR_NOT_UPLOADED"
    # cost(b) = pre_tile_us * Hq * sum over b's rows p of min(p + 1, L) / 128^2, L = 40:
    # blocks hold rows 0-15, 16-31 and 32-39 (the partial last block)
    cost = [float(x) for x in got[got.index("cost") + 1:got.index("cost") + 4]]
    for c, keys in zip(cost, (sum(range(1, 17)), sum(range(17, 33)), sum(range(33, 41)))):
        assert c == pytest.approx(1.0 * 8 * keys / 16384, rel=1e-15)

    # prefix reading: each block's cost is its own hole cost plus every later one
    # (a suffix sum), so it falls with position; scored on cost alone (alpha 0,
    # beta 1) the block evicted is the last one
    pre = lines[1].split()
    cost_prefix = [float(x) for x in pre[pre.index("cost_prefix") + 1:pre.index("cost_prefix") + 4]]
    for b in range(3):
        assert cost_prefix[b] == pytest.approx(sum(cost[b:]), rel=1e-12)
    assert pre[pre.index("evict_prefix") + 1] == "2"
    # chunk chooser: candidates 128, 256 and the whole remainder 300; the choice
    # has the least predicted time per prefill token; a budget below every
    # candidate's time returns the smallest candidate, flagged outside the budget
    ch = lines[2].split()
    cv = dict(zip(ch[0:16:2], ch[1:16:2]))
    rest = ch[ch.index("cands") + 1:]
    cands = [int(x) for x in rest[0::2]]
    times = [float(x) for x in rest[1::2]]
    assert cands == [128, 256, 300] and cv["ncand"] == "3"
    per_tok = [t / c for c, t in zip(cands, times)]
    best = min(range(3), key=lambda i: (per_tok[i], -cands[i]))
    assert int(cv["chunk"]) == cands[best] and int(cv["tokens"]) == cands[best] and cv["within"] == "1"
    assert float(cv["time"]) == times[best] and float(cv["upt"]) == pytest.approx(per_tok[best], rel=1e-15)
    assert cv["tight_chunk"] == "128" and cv["tight_within"] == "0"
