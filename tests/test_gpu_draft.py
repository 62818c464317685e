"""The layer-skip draft step against the oracle's forward over the same plan.

The draft (MLX self-speculation post, "Code -> the implementation"; LayerSkip
summary, 4.3.1) runs the kept layers only, on its own KV cache whose slot s
holds layer plan[s].  Lossless self-speculation says nothing about what the
draft computes, so these tests compare the draft itself: its logits and
token (spec_draft_step_logits) with orc.forward over the same plan, every
draft cache slot with the oracle's draft cache (before and after a draft
rollback), and, over whole self-speculative runs, the drafted tokens and
accept lengths with the oracle's own self-speculative loop.  Plans: middle
skips of 25% and 50%, and non-contiguous ones, so that slot s != layer s.

Tolerances as in gpu_common: logits within 2e-2 abs + 2e-2 rel; tokens
exact unless the oracle's top-two margin is below 1e-3 (flagged)."""
import numpy as np
import pytest

import oracle
import synth
from conftest import small_gqa_cfg
from gpu_common import ATOL, RTOL, TIE_GAP, argmax_mismatches, assert_logits_close, make_model, torch_cuda

pytestmark = pytest.mark.gpu


def _cfg(name):
    """The tiny model (4 layers, MHA) and a 6-layer variant of the small GQA
    model, deep enough that 25% and 50% middle skips keep layer 0."""
    return synth.tiny() if name == "tiny" else synth.scaled(small_gqa_cfg(), n_layers=6)


def _plans(cfg):
    """Middle skips of 25% and 50% (tiny: [0,2,3] and [0,3]; 6 layers:
    [0,1,4,5] and [0,4,5]) and a plan with two separate gaps."""
    L = cfg.n_layers
    plans = {"skip25": oracle.layer_skip_plan(L, 0.25), "skip50": oracle.layer_skip_plan(L, 0.5)}
    plans["noncontig"] = [0, 1, 3] if L == 4 else [0, 2, 3, 5]
    return plans


CASES = [(c, p) for c in ("tiny", "gqa-small") for p in ("skip25", "skip50", "noncontig")]


def _compare_draft_cache(m, dc, cfg, plan, length, what):
    for si in range(len(plan)):
        k, v = m.kv_export(1, si, length)
        kr = dc.read(si, 0, length).reshape(length, cfg.n_kv_heads, cfg.head_dim)
        vr = dc.read(si, 1, length).reshape(length, cfg.n_kv_heads, cfg.head_dim)
        kg, vg = synth.bf16_to_f32(k), synth.bf16_to_f32(v)
        assert np.allclose(kg, kr, atol=ATOL, rtol=RTOL), (what, "K", si, float(np.abs(kg - kr).max()))
        assert np.allclose(vg, vr, atol=ATOL, rtol=RTOL), (what, "V", si, float(np.abs(vg - vr).max()))


@pytest.mark.parametrize("cfgname,planname", CASES)
def test_draft_step_logits_token_and_cache_match_oracle(cfgname, planname):
    torch = torch_cuda()
    import speculative_decoding_verify_pass_gb300 as sv
    cfg = _cfg(cfgname)
    plan = _plans(cfg)[planname]
    w = synth.make_weights(cfg)
    m = make_model(cfg, w, draft_plan=plan)
    orc = oracle.Oracle(cfg, w)
    p = synth.prompt(cfg, 80, stream=21)
    P = 37                                            # prefill length (off the 64-position page)
    m.prefill(p[:P])
    dc = orc.new_cache(len(plan))
    orc.forward(dc, plan, p[:P], 0, logits_from=None)
    _compare_draft_cache(m, dc, cfg, plan, P, "after prefill")

    pos = P
    # n = 1 steps, then a catch-up pair (n = 2), then a rollback of the draft
    # cache by two positions and a re-fed pair, then two more single steps
    feeds = [[int(p[pos])], [int(p[pos + 1])], [int(p[pos + 2]), int(p[pos + 3])]]
    for step, feed in enumerate(feeds + ["rollback", [5, 6], [7], [int(p[50])]]):
        if feed == "rollback":
            pos -= 2
            m.rollback(sv.SPEC_CACHE_DRAFT, pos)
            dc.truncate(pos)
            continue
        tok, lg = m.draft_step(torch.tensor(feed, dtype=torch.int32, device="cuda"), logits=True)
        ref, _, _ = orc.forward(dc, plan, feed, pos, logits_from=0)
        what = "%s %s step %d (n=%d at %d)" % (cfgname, planname, step, len(feed), pos)
        assert_logits_close(lg.cpu().numpy(), ref, what)
        argmax_mismatches([int(tok.item())], ref[-1:])
        pos += len(feed)
        assert m.kv_len(sv.SPEC_CACHE_DRAFT) == pos
        _compare_draft_cache(m, dc, cfg, plan, pos, what)
    m.check_error()
    m.close()


def _selfspec_lockstep(torch, m, orc, plan, prompt, max_new, gamma):
    """The self-speculative loop run on the GPU and on the oracle side by
    side: every draft token and every verify row is compared, and a draft
    token that differs only inside a near tie is replaced by the oracle's
    on both sides, so that the runs keep the same inputs.  Returns (tokens,
    accept lengths, flagged near ties)."""
    import speculative_decoding_verify_pass_gb300 as sv
    full = orc.full_plan
    tc, dc = orc.new_cache(len(full)), orc.new_cache(len(plan))
    prompt = [int(t) for t in prompt]
    lg_t, _, _ = orc.forward(tc, full, prompt, 0, logits_from=len(prompt) - 1)
    orc.forward(dc, plan, prompt, 0, logits_from=None)
    y = int(m.prefill(prompt).item())
    flagged = len(argmax_mismatches([y], lg_t[-1:]))
    y = oracle.argmax(lg_t[-1])
    out, seq, accepts = [y], prompt + [y], []
    dlen = len(prompt)
    while len(out) < max_new:
        pos = len(seq) - 1
        feed = seq[dlen:pos + 1]
        drafts = []
        for _ in range(gamma):
            tok, lg = m.draft_step(torch.tensor(feed, dtype=torch.int32, device="cuda"), logits=True)
            ref, _, _ = orc.forward(dc, plan, feed, dlen, logits_from=len(feed) - 1)
            assert_logits_close(lg[-1:].cpu().numpy(), ref, "draft at %d" % dlen)
            flagged += len(argmax_mismatches([int(tok.item())], ref))
            d = oracle.argmax(ref[-1])
            dlen += len(feed)
            drafts.append(d)
            feed = [d]
        block = [seq[pos]] + drafts
        am, acc, lg, _ = m.verify(torch.tensor(block, dtype=torch.int32, device="cuda"), logits=True)
        ref, _, _ = orc.forward(tc, full, block, pos, logits_from=0)
        assert_logits_close(lg.cpu().numpy(), ref, "verify at %d" % pos)
        near = argmax_mismatches(am.cpu().numpy(), ref)
        flagged += len(near)
        a = [oracle.argmax(r) for r in ref]
        k = oracle.accept_len(block, a)
        if not near:
            assert int(acc.item()) == k
        accepts.append(k)
        emitted = drafts[:k] + [a[k]]
        out += emitted
        seq += emitted
        m.rollback(sv.SPEC_CACHE_TARGET, pos + k + 1)
        tc.truncate(pos + k + 1)
        dlen = min(pos + k + 1, dlen)
        m.rollback(sv.SPEC_CACHE_DRAFT, dlen)
        dc.truncate(dlen)
    return out[:max_new], accepts, flagged


@pytest.mark.parametrize("cfgname,planname,gamma", [("tiny", "skip50", 4), ("tiny", "noncontig", 3),
                                                    ("gqa-small", "skip25", 2), ("gqa-small", "noncontig", 5)])
def test_selfspec_drafts_and_accept_lengths_match_oracle(cfgname, planname, gamma):
    """Every draft token, verify row and accept length of a self-speculative
    run against the oracle's; the emitted tokens must also be the oracle's
    own self-speculative output and its plain greedy output."""
    torch = torch_cuda()
    cfg = _cfg(cfgname)
    plan = _plans(cfg)[planname]
    w = synth.make_weights(cfg)
    m = make_model(cfg, w, draft_plan=plan)
    orc = oracle.Oracle(cfg, w)
    prompt = synth.prompt(cfg, 40, stream=23)
    got, accepts, flagged = _selfspec_lockstep(torch, m, orc, plan, prompt, 40, gamma)
    want, want_acc = oracle.selfspec_generate(orc, plan, prompt, 40, gamma)
    if not flagged:
        assert got == want and accepts == want_acc
        assert got == oracle.greedy_generate(orc, prompt, 40)
    m.check_error()
    m.close()


def test_full_plan_draft_logits_equal_verify_rows_bitwise():
    """With every layer kept, a draft step is the verify pass's arithmetic
    on the draft cache: its logits equal the target's verify row of the same
    token at the same position, bit for bit (batch invariance)."""
    torch = torch_cuda()
    cfg = small_gqa_cfg()
    w = synth.make_weights(cfg)
    m = make_model(cfg, w, draft_plan=list(range(cfg.n_layers)))
    p = synth.prompt(cfg, 60, stream=24)
    m.prefill(p[:45])
    for j in range(3):
        blk = torch.tensor([int(p[45 + j])], dtype=torch.int32, device="cuda")
        tok, lg_d = m.draft_step(blk, logits=True)
        am, _, lg_v, _ = m.verify(blk.clone(), logits=True)
        assert torch.equal(lg_d, lg_v), j
        assert int(tok.item()) == int(am[0].item())
    m.close()
