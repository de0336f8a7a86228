"""The bench's algorithmic byte count (no GPU), written out by hand for the
32-layer workload's heads: 8 kv heads, 32 query heads, d = 128, bf16."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from demand_paged_kv_gqa_b300 import synth  # noqa: E402


def test_attention_bytes_by_hand():
    w = synth.WORKLOADS["llama8b_32layer"]
    # one request-layer with 1000 resident tokens, not at a boundary
    kv = 1000 * (8 * 128 * 2) * 2                    # K and V rows, bf16
    fixed = (32 * 128 * 2) * 2 + (8 * 128 * 2) * 2 * 2 + (8 * 128 * 4) * 2 * 2
    assert fixed == 40960
    bt = 1000 / 16 * 4
    assert bench.attention_bytes(w, 1000, 1, 0) == kv + fixed + bt
    # at a boundary both summaries' fp32 scores are written for every resident key
    assert bench.attention_bytes(w, 1000, 1, 1000) - bench.attention_bytes(w, 1000, 1, 0) == 1000 * 2 * 8 * 4


def test_reference_arm_line_on_cpu():
    # the oracle arm runs on the host cores and prints the contract's line
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    for k in ("metric", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "dtype", "config"):
        assert k in line


def test_timed_regions_run_without_garbage_collection():
    # the collector is off inside a timed region and back on after it, also
    # when the region raises
    import gc
    assert gc.isenabled()
    with bench.no_gc():
        assert not gc.isenabled()
    assert gc.isenabled()
    try:
        with bench.no_gc():
            raise ValueError("inside a timed region")
    except ValueError:
        pass
    assert gc.isenabled()
