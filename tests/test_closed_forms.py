"""Pins of the step-time model's closed forms (MoE speculative-decoding page).

Monte Carlo over the seeded generators, exact counts of generated tensors and
algebraic identities; no check reuses the formula it tests."""
import math

import numpy as np
import pytest

import synth
from conftest import small_gqa_cfg, small_moe_cfg
from oracle import closed_forms as cf


@pytest.mark.parametrize("n", [1, 2, 3, 5, 8])
def test_expected_union_matches_monte_carlo(n):
    E, k = 64, 6
    draws = 20000
    tr = synth.routing_trace(1, n * (draws // n + 1), E, k, stream=n)[0]
    sizes = []
    # independent windows: restart the chain every n tokens by only using windows
    # whose first token drew a fresh set; the trace's first token is always fresh
    for start in range(0, tr.shape[0] - n, n):
        sizes.append(len(set(tr[start:start + n].ravel().tolist())))
    sizes = np.array(sizes, dtype=np.float64)
    want = cf.expected_union(n, E, k)
    # windows after the first start mid-chain: their first set is still a
    # uniform k-subset (fresh or copied from a uniform one), so the law holds
    se = sizes.std(ddof=1) / math.sqrt(len(sizes))
    assert abs(sizes.mean() - want) < 4 * se + 1e-9, (sizes.mean(), want)
    if n == 1:
        assert want == k
    assert want <= min(E, n * k)


def test_routing_trace_structure():
    tr = synth.routing_trace(3, 400, 64, 6)
    assert tr.shape == (3, 400, 6)
    reuse = np.mean([np.array_equal(tr[0, t], tr[0, t - 1]) for t in range(1, 400)])
    assert 0.4 < reuse < 0.6
    for l in range(3):
        for t in range(400):
            assert len(set(tr[l, t].tolist())) == 6


@pytest.mark.parametrize("alpha", [0.0, 0.3, 0.5, 0.7, 0.9, 1.0])
@pytest.mark.parametrize("gamma", [1, 2, 4, 7, 15])
def test_expected_tokens_matches_geometric_draws(alpha, gamma):
    acc = synth.geometric_accept_lengths(20000, alpha, gamma, stream=gamma)
    emitted = acc + 1
    want = cf.expected_tokens(alpha, gamma)
    if alpha in (0.0, 1.0):
        assert np.all(emitted == (1 if alpha == 0.0 else gamma + 1))
        assert want == (1 if alpha == 0.0 else gamma + 1)
    else:
        se = emitted.std(ddof=1) / math.sqrt(len(emitted))
        assert abs(emitted.mean() - want) < 4 * se
        assert abs(want - (1 - alpha ** (gamma + 1)) / (1 - alpha)) < 1e-12   # geometric sum


def test_draft_corruption_acceptance_is_geometric():
    truth = synth.uniform_ints(16 * 4000, 0, 1000, 9, 9)
    for alpha in (0.5, 0.9):
        d = synth.corrupt_drafts(truth, alpha, 1000, stream=int(alpha * 10))
        ok = (d == truth).reshape(4000, 16)
        assert abs(ok.mean() - alpha) < 0.01
        run = np.array([next((j for j in range(16) if not r[j]), 16) for r in ok])
        for j in (1, 2, 4):
            assert abs(np.mean(run >= j) - alpha ** j) < 0.03
        assert np.all((d == truth) | (d != truth))
        assert np.all(d[~(d == truth)] != truth[~(d == truth)])


def test_dedup_criterion_is_the_time_comparison():
    rng = np.random.default_rng(5)
    for _ in range(1000):
        bytes_ps = rng.uniform(1e8, 1e10)
        bytes_dd = bytes_ps * rng.uniform(0.05, 1.0)
        bw_ps = rng.uniform(1e11, 8e12)
        bw_dd = bw_ps * rng.uniform(0.2, 1.2)
        faster = bytes_dd / bw_dd < bytes_ps / bw_ps
        assert cf.dedup_faster(bytes_dd / bytes_ps, bw_dd / bw_ps) == faster
    assert cf.crossover([0.9, 0.7, 0.5, 0.4], [0.5, 0.6, 0.6, 0.6], [1, 2, 3, 4]) == 3
    assert cf.crossover([0.9, 0.8], [0.3, 0.3], [1, 2]) is None


def test_best_draft_length_is_a_monotone_staircase():
    """gamma*(alpha) never decreases as alpha grows, for verify times that grow
    with the block (the staircase of the MoE page), over the 22 alpha values."""
    alphas = np.linspace(0.0, 1.0, 22)
    for t_draft in (0.0, 0.05, 0.2):
        for slope in (0.01, 0.05, 0.2):
            tv = lambda n: 1.0 + slope * (n - 1) + 0.002 * (n - 1) ** 2
            g = [cf.best_draft_length(a, tv, t_draft, range(0, 16)) for a in alphas]
            assert all(b >= a for a, b in zip(g, g[1:])), (t_draft, slope, g)
            assert g[0] == 0


def test_speculation_condition():
    # alpha = 0: one token per cycle, so speculation only wins if the cycle is cheaper
    assert not cf.speculation_wins(0.0, 3, 1.0, 1.05, 0.1)
    assert cf.speculation_wins(0.9, 3, 1.0, 1.05, 0.1)
    # break-even: E[tau] * T1 == T_cycle is not a win
    assert not cf.speculation_wins(1.0, 1, 1.0, 1.5, 0.5)


@pytest.mark.parametrize("make", ["tiny", "gqa", "moe"])
def test_pass_bytes_counts_every_generated_weight(make):
    cfg = {"tiny": synth.tiny(), "gqa": small_gqa_cfg(), "moe": small_moe_cfg()}[make]
    w = synth.make_weights(cfg)
    mats = 0
    for L in w.layers:
        for key, val in L.items():
            if key.endswith("norm"):
                continue
            for t in (val if isinstance(val, list) else [val]):
                mats += t.nbytes
    n, ctx = 5, 33
    b = cf.pass_bytes(cfg, n, ctx, unique_experts_per_layer=cfg.n_experts if cfg.n_experts else None)
    weights = b.qkv + b.o + b.ffn_dense + b.router + b.experts + b.shared
    assert weights == mats                           # every expert counted once when |U| = E
    assert b.lm_head == w.lm_head_or_embed().nbytes
    kvw = cfg.n_kv_heads * cfg.head_dim
    assert b.kv_read == cfg.n_layers * 2 * kvw * ctx * 2
    assert b.kv_write == cfg.n_layers * 2 * kvw * n * 2
    if cfg.n_experts:
        per_expert = sum(t.nbytes for t in (w.layers[1]["e_gate"][0], w.layers[1]["e_up"][0], w.layers[1]["e_down"][0]))
        assert b.experts_per_slot == (cfg.n_layers - 1) * n * cfg.top_k * per_expert


def test_pass_bytes_of_the_workload_shapes():
    """Analytic bytes of the big shapes, from their matrix dimensions."""
    q4 = synth.qwen3_4b()
    b = cf.pass_bytes(q4, 4, 2048)
    per_layer = (6144 * 2560 + 2560 * 4096 + 3 * 9728 * 2560) * 2
    assert b.qkv + b.o + b.ffn_dense == 36 * per_layer
    assert b.lm_head == 151936 * 2560 * 2
    assert abs(b.total / 1e9 - 8.347) < 0.01
    moe = synth.moe_v2lite()
    per_expert = 3 * 1408 * 2048 * 2
    assert abs(per_expert / 1e6 - 17.30) < 0.01
