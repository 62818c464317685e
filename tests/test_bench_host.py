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
    q = out["qkv"]
    assert (q["launches"], q["ready_to_exit"], q["work_to_exit"], q["gap"]) == (2, 4.0, 1.25, 1.0)
    assert q["ready_spread"] == 0.05            # (100 + 0) / 2 launches
    assert q["cta_ready_to_work_med"] == 2.6    # medians 3.2 and 2.0
    assert q["cta_ready_to_work_max"] == 2.7    # maxima 3.4 and 2.0
    assert q["work_spread"] == 0.25             # (500 + 0) / 2
    a = out["attn_partial"]
    assert (a["launches"], a["ready_to_exit"], a["work_to_exit"], a["gap"]) == (1, 1.0, 0.0, 1.0)


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


def _stamp(t):
    import datetime
    return datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]


def test_clock_summary_keeps_only_samples_taken_inside_the_timed_region():
    t0 = 1_800_000_000.0
    line = "{ts}, {sm}, 2070, 900.5, {hw}, Not Active, Not Active, {cap}"
    rows = [(-0.1, 1200, "Not Active", "Not Active"),   # before the region
            (0.1, 2070, "Not Active", "Active"),
            (0.2, 2040, "Not Active", "Not Active"),
            (0.3, 2070, "Not Active", "Not Active"),
            (1.0, 900, "Active", "Not Active")]          # long after it
    # every line read only at the end (a buffered pipe): the samples' own stamps decide
    lines = [(t0 + 5.0, line.format(ts=_stamp(t0 + dt), sm=sm, hw=hw, cap=cap)) for dt, sm, hw, cap in rows]
    lines.append((t0 + 5.0, "garbled"))
    out = bench.summarize_clock_lines(lines, t0, t0 + 0.25, slack=0.1)
    assert out == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_summary_uses_arrival_time_without_a_stamp_and_falls_back_to_every_sample():
    line = "n/a, 2070, 2070, 900.5, Not Active, Not Active, Not Active, Not Active"
    out = bench.summarize_clock_lines([(1.1, line), (1.15, line), (3.0, line)], 1.0, 1.2)
    assert out["samples"] == 2 and "note" not in out
    out = bench.summarize_clock_lines([(5.0, line), (5.1, line)], 1.0, 1.2)
    assert out["samples"] == 2 and out["sm_mhz"] == 2070.0 and "note" in out
    assert bench.summarize_clock_lines([], 1.0, 1.2)["sm_mhz"] is None


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) on the tiny
    shape: one JSON line with the contract's keys, its own cpu_baseline and
    an e2e entry that moves no bytes."""
    import json
    import subprocess
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                          "--ctx", "128", "--steps", "2", "--warmup", "3"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tok/s"
    assert d["steps"] == 2 and d["warmup"] == 3 and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_geometric_schedule_accepts_the_clean_prefix_and_advances():
    """The cycle schedule of the default workload: each cycle's accept length
    is its number of leading clean drafts (corrupted drafts differ from the
    truth), the next block starts accept+1 positions later, and over many
    cycles P(accept >= j) follows alpha^j."""
    import synth
    n, alpha, V = 8, 0.7, 128256
    sched = bench.geometric_schedule(n, alpha, 4000, V)
    assert sched[0][0] == 0
    for (j0, k0), (j1, _) in zip(sched, sched[1:]):
        assert 0 <= k0 <= n - 1 and j1 == j0 + k0 + 1
    ks = np.array([k for _, k in sched])
    for j in range(1, n):
        p = alpha ** j
        assert abs(np.mean(ks >= j) - p) < 4 * np.sqrt(p * (1 - p) / len(ks)) + 1e-9, j
    greedy = list(synth.prompt(synth.llama31_8b(), sched[40][0] + n + 1, stream=3))
    blocks = bench.geometric_blocks(greedy, sched[:40], n, alpha, V)
    for s, (j, k) in enumerate(sched[:40]):
        assert blocks[s, 0] == greedy[j]
        assert list(blocks[s, 1:k + 1]) == greedy[j + 1:j + k + 1]
        if k < n - 1:
            assert blocks[s, k + 1] != greedy[j + k + 1]


def test_launch_segments_tile_the_pass():
    st = _stamps([
        [(0, 1000, 2000, 5000, 6000), (1, 1100, 2100, 5500, 7000)],   # first launch: from its first entry
        [(0, 6500, 8000, 0, 9000)],                                     # starts before the previous exit
        [],                                                             # nothing recorded
        [(3, 9100, 10000, 12000, 13000)],
    ])
    segs = bench.launch_segments(st, [0, 16, 1, 3])
    assert segs == [(0, 6.0), (16, 2.0), (3, 4.0)]
    assert sum(t for _, t in segs) == (13000 - 1000) / 1e3
