"""Host-side logic of the benchmark suites, on CPU: the launch-trace
breakdown (per launch kind: inputs ready to last exit, last main-work stamp
to exit, gap after the previous launch)."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _stamps(launches):
    """[ctas][launches][4] from {launch: [(cta, entry, ready, work, exit)]}."""
    st = np.zeros((512, len(launches), 4), dtype=np.int64)
    for l, rows in enumerate(launches):
        for cta, *v in rows:
            st[cta, l] = v
    return st


def test_trace_breakdown_per_kind():
    st = _stamps([
        [(0, 1000, 2000, 5000, 6000), (1, 1100, 2100, 5500, 7000)],   # QKV
        [(0, 6500, 8000, 0, 9000)],                                     # attention partials
        [(3, 9100, 10000, 12000, 13000)],                               # QKV again
    ])
    out, span = bench.trace_breakdown(st, [0, 16, 0])
    assert span == 12.0
    assert out["qkv"] == {"launches": 2, "ready_to_exit": 4.0, "work_to_exit": 1.25, "gap": 1.0}
    assert out["attn_partial"] == {"launches": 1, "ready_to_exit": 1.0, "work_to_exit": 0.0, "gap": 1.0}


def test_trace_breakdown_skips_launches_without_live_ctas_and_uses_entry_when_never_waited():
    st = _stamps([
        [(0, 1000, 0, 0, 3000)],          # embedding: no dependency-wait stamp
        [],                               # a launch that recorded nothing
        [(5, 3500, 4000, 0, 4500)],
    ])
    out, span = bench.trace_breakdown(st, [18, 1, 17])
    assert set(out) == {"embed", "attn_merge"}
    assert out["embed"]["ready_to_exit"] == 2.0
    assert out["attn_merge"]["gap"] == 1.0
    assert span == 3.5
