"""Shared prefix cache (LayerSkip summary, 4.3.3 "Single KV Cache"): the
draft's leading layers use the target's KV cache.

Self-speculative decoding must stay lossless (equal to plain greedy), give
the same drafts, accept lengths and final target cache, bit for bit, as
with separate caches, and the draft's shared slots must be the target's own
pools.  The emitted tokens and accept lengths are also checked against the
oracle's plain greedy decoding and its own self-speculative loop over the
same plan (exact, unless the oracle's greedy run passes a near tie)."""
import numpy as np
import pytest

import oracle
import synth
from conftest import small_gqa_cfg
from gpu_common import TIE_GAP, make_model, torch_cuda


def _oracle_greedy_with_margin(orc, prompt, max_new):
    """The oracle's plain greedy tokens and the smallest top-two logit margin
    met on the way (below TIE_GAP the GPU may take the other token)."""
    cache = orc.new_cache()
    lg, _, _ = orc.forward(cache, orc.full_plan, prompt, 0, logits_from=len(prompt) - 1)
    out, margin = [], np.inf
    while True:
        row = np.sort(lg[-1])
        margin = min(margin, float(row[-1] - row[-2]))
        out.append(oracle.argmax(lg[-1]))
        if len(out) == max_new:
            return out, margin
        lg, _, _ = orc.forward(cache, orc.full_plan, [out[-1]], cache.len, logits_from=0)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfgname,frac,gamma", [("tiny", 0.5, 4), ("tiny", 0.25, 2), ("gqa-small", 0.34, 3),
                                                ("tiny", 0.0, 5)])
def test_shared_prefix_selfspec_is_lossless_and_equals_separate_caches(cfgname, frac, gamma):
    torch_cuda()
    cfg = synth.tiny() if cfgname == "tiny" else small_gqa_cfg()
    w = synth.make_weights(cfg)
    plan = list(range(cfg.n_layers)) if frac == 0.0 else oracle.layer_skip_plan(cfg.n_layers, frac)
    prompt = synth.prompt(cfg, 40, stream=3)
    runs = {}
    for share in (False, True):
        m = make_model(cfg, w, draft_plan=plan)
        if share:
            m.share_prefix(True)
        out, acc = m.selfspec(prompt, 48, gamma)
        m.check_error()
        n_pos = m.kv_len(0)
        kv = [m.kv_export(0, l, n_pos) for l in range(cfg.n_layers)]
        runs[share] = (out, acc, n_pos, kv)
        if share:
            shared = 0
            while shared < len(plan) and plan[shared] == shared:
                shared += 1
            dl = m.kv_len(1)
            for si in range(shared):      # the draft's shared slots are the target's layers
                dk, dv = m.kv_export(1, si, dl)
                tk, tv = m.kv_export(0, si, dl)
                assert np.array_equal(dk, tk) and np.array_equal(dv, tv)
        m.close()
    g = make_model(cfg, w)
    greedy = g.greedy(prompt, 48)
    g.close()
    (oa, aa, na, kva), (ob, ab, nb, kvb) = runs[False], runs[True]
    assert ob == greedy and oa == greedy
    orc = oracle.Oracle(cfg, w)
    want, margin = _oracle_greedy_with_margin(orc, prompt, 48)
    if margin >= TIE_GAP:
        assert ob == want
        want_ss, want_acc = oracle.selfspec_generate(orc, plan, prompt, 48, gamma)
        assert want_ss == want and ab == want_acc
    assert ab == aa and nb == na
    for l in range(cfg.n_layers):
        assert np.array_equal(kva[l][0], kvb[l][0]) and np.array_equal(kva[l][1], kvb[l][1]), l
    if frac == 0.0:
        assert all(k == gamma for k in ab)


def test_share_prefix_needs_a_draft_plan():
    torch_cuda()
    import speculative_decoding_verify_pass_gb300 as sv
    cfg = synth.tiny()
    m = make_model(cfg, synth.make_weights(cfg))
    with pytest.raises(sv.SpecError) as e:
        m.share_prefix(True)
    assert e.value.status == sv.SPEC_ERR_STATE
    m.close()
