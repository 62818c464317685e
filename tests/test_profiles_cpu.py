"""The byte model against the committed counter captures, on CPU.

"Speculative Decoding for Mixture-of-Experts Models: Expert Bytes, Kernel
Bandwidth and the Best Draft Length" (abstract) models a step as the bytes
each kernel requests over that kernel's bandwidth.  The oracle's closed forms
count those bytes; the ncu summaries under profiles/ hold what DRAM and L2
actually served for the same launches.  These tests read the summaries as
data and check them against the closed forms:
- every dense GEMM kind reads its weight bytes from DRAM once (within 1%);
- a deduplicating expert launch reads each distinct expert, and each shared
  expert, from DRAM once (within 1%);
- a per-slot expert launch requests one expert per (token, slot): its L2 read
  volume over the dedup launch's follows the analytic read ratio.
"""
import os
import re

import pytest

import synth
from oracle import closed_forms

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROFILES = os.path.join(ROOT, "profiles")


def _gemm_traffic():
    path = os.path.join(PROFILES, "gemm_kernel_dram_llama-3.1-8b.txt")
    kinds = {}
    for line in open(path):
        f = line.split()
        if len(f) == 6 and f[0] == "kind":
            kinds[int(f[1])] = (int(f[3]), int(f[5]))
    return kinds


def test_dense_gemm_kinds_read_their_weights_once():
    cfg = synth.llama31_8b()
    one_layer = closed_forms.pass_bytes(cfg, 1, 0, plan=[0])
    weights = {
        0: one_layer.qkv,
        1: (one_layer.o + one_layer.ffn_dense // 3) / 2,   # mean of O and down, as the capture averages them
        2: 2 * one_layer.ffn_dense // 3,                    # gate and up
        3: one_layer.lm_head,
    }
    kinds = _gemm_traffic()
    assert set(kinds) == set(weights)
    for k, (read, write) in kinds.items():
        assert 1.0 <= read / weights[k] < 1.01, (k, read, weights[k])
        assert write < 0.01 * weights[k]


def _moe_rows():
    path = os.path.join(PROFILES, "moe_expert_bytes_moe-v2-lite_n8.md")
    rows = []
    mb = lambda x: float(x.replace("MB", "").strip()) * 1e6
    for line in open(path):
        if not re.match(r"\| (per_slot|dedup) \|", line):
            continue
        c = [x.strip() for x in line.strip().strip("|").split("|")]
        rows.append({"mode": c[0], "layer": int(c[1]), "kind": c[2], "reads": int(c[3]), "unique": int(c[4]),
                     "requested": mb(c[5]), "unique_bytes": mb(c[6]), "dram": mb(c[7]), "l2": mb(c[9])})
    return rows


def test_moe_expert_bytes_follow_the_byte_model():
    cfg = synth.moe_v2lite()
    per_expert = closed_forms.pass_bytes(cfg, 1, 0, plan=[cfg.first_moe_layer], unique_experts_per_layer=1).experts
    part = {"gate-up": 2 * per_expert / 3, "down": per_expert / 3}
    rows = _moe_rows()
    assert len(rows) == 8
    for r in rows:
        # the table's analytic columns are the closed form's expert bytes (0.1 MB rounding)
        assert r["requested"] == pytest.approx(r["reads"] * part[r["kind"]], abs=0.06e6)
        assert r["unique_bytes"] == pytest.approx(r["unique"] * part[r["kind"]], abs=0.06e6)
        assert r["reads"] == (8 * cfg.top_k + cfg.n_shared_experts if r["mode"] == "per_slot" else r["unique"])
        if r["mode"] == "dedup":
            assert 1.0 <= r["dram"] / r["unique_bytes"] < 1.01, r
        else:
            assert r["dram"] >= r["unique_bytes"]             # repeats are served from L2, never fewer reads
    by = {(r["mode"], r["layer"], r["kind"]): r for r in rows}
    for (mode, layer, kind), ps in by.items():
        if mode != "per_slot":
            continue
        dd = by[("dedup", layer, kind)]
        analytic = ps["reads"] / dd["reads"]
        assert 0.85 * analytic <= ps["l2"] / dd["l2"] <= 1.05 * analytic, (layer, kind)
