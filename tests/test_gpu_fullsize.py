"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times: one verify pass over every layer of the Qwen3-4B-,
Llama-3.1-8B-, Qwen3-8B- and DeepSeek-V2-Lite-shaped models at their
benchmark contexts (seeded synthetic KV), plus full-width one-layer cases;
every logit row is compared with the oracle computing the same pass on the
same weights.

The reference is the oracle's fp64-accumulating build.  Each case's bound
comes from tests/golden/fullsize_floor.txt, the fp32 oracle's own deviation
from that build on the same inputs: where that floor is inside the stated
logit tolerance the tolerance holds as stated; elsewhere the GPU may deviate
at most FLOOR_FACTOR times as much as the fp32 oracle does (gpu_common)."""
import gc
import importlib.util
import os

import numpy as np
import pytest

import oracle
import synth
from gpu_common import (FLOOR_FACTOR, TIE_GAP, argmax_mismatches, assert_within_floor, load_floor, make_model,
                        torch_cuda)

pytestmark = pytest.mark.gpu

_spec = importlib.util.spec_from_file_location(
    "make_fullsize_floor", os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                                        "make_fullsize_floor.py"))
_floor_script = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(_floor_script)

FLOOR = load_floor()
DENSE = [k for k, c in FLOOR.items() if c["preset"] != "moe-v2-lite"]
MOE = [k for k, c in FLOOR.items() if c["preset"] == "moe-v2-lite"]


def _config(c):
    return _floor_script.case_config(c["preset"], c["layers"], c["ctx"], c["n"])


def _tie_gap(c):
    """A near tie is a top-two margin the fp32 arithmetic itself may reorder:
    1e-3 where the floor is inside the tolerance, else twice the floor's
    largest logit deviation."""
    return TIE_GAP if c["share"] == 0.0 else max(TIE_GAP, 2.0 * c["max"])


def _load_context(m, cfg, ctx):
    for l in range(cfg.n_layers):
        m.kv_load(0, l, synth.synthetic_kv(cfg, l, ctx, 0), synth.synthetic_kv(cfg, l, ctx, 1))
    m.kv_set_len(0, ctx)


@pytest.mark.parametrize("case", DENSE)
def test_dense_fullsize_verify_matches_oracle(case):
    torch = torch_cuda()
    c = FLOOR[case]
    cfg = _config(c)
    w = synth.make_weights(cfg)
    m = make_model(cfg, w)
    _load_context(m, cfg, c["ctx"])
    toks = synth.prompt(cfg, c["n"], stream=c["stream"])
    am, acc, lg, _ = m.verify(torch.tensor(toks, dtype=torch.int32, device="cuda"), logits=True)
    m.check_error()
    am, acc, lg = am.cpu().numpy(), int(acc.item()), lg.cpu().numpy()
    m.close()
    del m
    gc.collect()
    o64 = oracle.Oracle(cfg, w, acc64=True)
    oc = o64.new_cache()
    _floor_script.load_context(o64, oc, cfg, c["ctx"])
    ref, _, _ = o64.forward(oc, o64.full_plan, toks, c["ctx"])
    assert_within_floor(lg, ref, c, case)
    flagged = argmax_mismatches(am, ref, tie_gap=_tie_gap(c))
    if not flagged:
        assert acc == oracle.accept_len(toks, [int(np.argmax(r)) for r in ref])
    del o64, oc, w
    gc.collect()


@pytest.mark.parametrize("case", MOE)
def test_moe_fullsize_verify_matches_oracle_and_modes_agree(case):
    """n = 4, and n = 8 where deduplication reads fewest bytes relative to
    per-slot; both modes must give the same bits and match the oracle."""
    torch = torch_cuda()
    import speculative_decoding_verify_pass_gb300 as sv
    c = FLOOR[case]
    ctx, n = c["ctx"], c["n"]
    cfg = _config(c)
    w = synth.make_weights(cfg)
    m = make_model(cfg, w)
    _load_context(m, cfg, ctx)
    toks = synth.prompt(cfg, n, stream=c["stream"])
    out = {}
    for mode in (sv.SPEC_MOE_PER_SLOT, sv.SPEC_MOE_DEDUP):
        m.moe_mode(mode)
        m.kv_set_len(0, ctx)
        am, acc, lg, ids = m.verify(torch.tensor(toks, dtype=torch.int32, device="cuda"), logits=True,
                                    expert_ids=True)
        out[mode] = (am.cpu().numpy(), lg.cpu().numpy(), ids.cpu().numpy())
    m.check_error()
    m.close()
    del m
    gc.collect()
    ps, dd = out[sv.SPEC_MOE_PER_SLOT], out[sv.SPEC_MOE_DEDUP]
    for x, y in zip(ps, dd):
        assert np.array_equal(x, y)           # per-slot and dedup: bitwise equal
    gids = ps[2]
    o64 = oracle.Oracle(cfg, w, acc64=True)
    moe_layers = slice(cfg.first_moe_layer, cfg.n_layers)
    # free routing: routing is discontinuous, so once rounding drift flips one
    # choice the residuals part and later choices follow; the GPU may differ
    # from the fp64 oracle in at most FLOOR_FACTOR times as many slots as the
    # fp32 oracle does
    oc = o64.new_cache()
    _floor_script.load_context(o64, oc, cfg, ctx)
    _, ids_free, _ = o64.forward(oc, o64.full_plan, toks, ctx, logits_from=None, want_routing=True)
    mism = float(np.mean(ids_free[moe_layers] != gids[moe_layers]))
    assert mism <= FLOOR_FACTOR * c["route_mismatch"], "expert ids differ in %.2f%% of slots (fp32 oracle: %.2f%%)" % (
        100 * mism, 100 * c["route_mismatch"])
    # teacher-forced: with the oracle run on the GPU's routing, every GPU
    # choice must be the oracle's own top-k at that slot, unless the two
    # candidates' probabilities are closer than twice the largest router
    # probability drift between the fp32 and fp64 oracles
    oc.truncate(ctx)
    probs = np.zeros((cfg.n_layers, n, cfg.n_experts), np.float32)
    ref, _, _ = o64.forward(oc, o64.full_plan, toks, ctx, want_routing=True, forced_ids=np.maximum(gids, 0),
                            probs=probs)
    for l in range(cfg.first_moe_layer, cfg.n_layers):
        for i in range(n):
            pr = probs[l, i].astype(np.float64)
            top = sorted(range(cfg.n_experts), key=lambda e: (-pr[e], e))[:cfg.top_k]
            kth = min(pr[e] for e in top)
            for e in set(int(e) for e in gids[l, i]) - set(top):
                gap = kth - pr[e]
                assert gap < 2.0 * c["route_dp"], "layer %d token %d: GPU expert %d trails the oracle's top-%d by %.3g" % (
                    l, i, e, cfg.top_k, gap)
    assert_within_floor(ps[1], ref, c, "moe ctx=%d n=%d" % (ctx, n))
    argmax_mismatches(ps[0], ref, tie_gap=_tie_gap(c))
    del o64, oc, w
    gc.collect()
