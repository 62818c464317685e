"""Sampled verification on the GPU (spec_accept_sampled) against the oracle.

The rule is the standard one of speculative sampling (oracle/sampling.py;
LayerSkip summary 4.3.2 states its property: the output distribution is the
full model's).  Here:
- accept_len and the drawn token against the oracle on seeded random logits,
  at vocabularies of 1000 and 128256, for blocks of 1..16, exactly except
  where the oracle's own decision is within a near-tie margin (flagged);
- the first emitted token's distribution against the target's, by Monte
  Carlo through the GPU call;
- self-speculative decoding with sampling at a vanishing temperature equals
  plain greedy decoding;
- argument errors."""
import numpy as np
import pytest

import synth
from gpu_common import make_model, torch_cuda
from oracle import sampling as smp

pytestmark = pytest.mark.gpu

ACC_TIE = 1e-4     # log-domain margin of an accept test (fp32 logits/T, fp32 chunk sums)
DRAW_TIE = 1e-6    # margin of the draw, as a fraction of the total weight


def _model(vocab):
    cfg = synth.scaled(synth.tiny(), vocab=vocab)
    return make_model(cfg, synth.make_weights(cfg)), cfg


def _case(rng, V, n, T):
    tl = (rng.normal(size=(n, V)) * 2.0).astype(np.float32)
    dl = (tl[:max(n - 1, 0)] + rng.normal(size=(max(n - 1, 0), V)) * 0.8).astype(np.float32)
    x = [int(rng.integers(0, V))]
    for j in range(n - 1):
        x.append(smp.draw(smp.softmax_t(dl[j], T), rng.random()))
    u = rng.random(n)
    return tl, dl, x, u


@pytest.mark.parametrize("V,trials", [(1000, 240), (128256, 40)])
def test_accept_sampled_matches_oracle(V, trials):
    torch = torch_cuda()
    m, cfg = _model(V)
    rng = np.random.default_rng(V)
    flagged = 0
    for t in range(trials):
        n = int(rng.integers(1, 17))
        T = float(rng.choice([0.5, 1.0, 2.0]))
        tl, dl, x, u = _case(rng, V, n, T)
        k_o, tok_o = smp.accept_sampled(tl, dl, x, T, u[:n - 1], u[n - 1])
        dtl = torch.from_numpy(tl).to("cuda")
        ddl = torch.from_numpy(dl).to("cuda") if n > 1 else None
        blk = torch.tensor(x, dtype=torch.int32, device="cuda")
        k, tok = m.accept_sampled(dtl, ddl, blk, T, u)
        k, tok = int(k.item()), int(tok.item())
        if (k, tok) != (k_o, tok_o):
            am, dm = smp.decision_margins(tl, dl, x, T, u[:n - 1], u[n - 1])
            assert am < ACC_TIE or dm < DRAW_TIE, (t, n, T, (k, tok), (k_o, tok_o), am, dm)
            flagged += 1
    m.check_error()
    assert flagged <= max(1, trials // 50)
    m.close()


def test_first_emitted_token_follows_the_target_distribution():
    """Monte Carlo through the GPU call: one draft drawn from q, then the
    sampled accept; the first emitted token is distributed as p_0."""
    torch = torch_cuda()
    V = 8
    m, cfg = _model(V)
    rng = np.random.default_rng(21)
    tl = (rng.normal(size=(2, V)) * 1.5).astype(np.float32)
    dl = (tl[:1] + rng.normal(size=(1, V)) * 1.2).astype(np.float32)
    p0 = smp.softmax_t(tl[0], 1.0)
    q0 = smp.softmax_t(dl[0], 1.0)
    dtl, ddl = torch.from_numpy(tl).to("cuda"), torch.from_numpy(dl).to("cuda")
    trials = 6000
    draws = rng.random((trials, 3))
    blk = torch.zeros((trials, 2), dtype=torch.int32, device="cuda")
    blk[:, 1] = torch.tensor([smp.draw(q0, d[0]) for d in draws], dtype=torch.int32)
    us = torch.from_numpy(draws[:, 1:].copy()).to("cuda")
    acc = torch.zeros(trials, dtype=torch.int32, device="cuda")
    tok = torch.zeros(trials, dtype=torch.int32, device="cuda")
    import speculative_decoding_verify_pass_gb300 as sv
    for i in range(trials):
        sv.spec_accept_sampled(m.h, dtl, ddl, blk[i], 1.0, us[i], acc[i:i + 1], tok[i:i + 1])
    acc, tok, x1 = acc.cpu().numpy(), tok.cpu().numpy(), blk[:, 1].cpu().numpy()
    first = np.where(acc == 1, x1, tok)
    counts = np.bincount(first, minlength=V).astype(np.float64)
    dev = np.abs(counts - trials * p0)
    assert np.all(dev <= 4.5 * np.sqrt(trials * p0 * (1 - p0)) + 1e-9), (counts / trials, p0)
    m.close()


def test_vanishing_temperature_selfspec_equals_greedy():
    torch_cuda()
    import speculative_decoding_verify_pass_gb300 as sv
    cfg = synth.tiny()
    w = synth.make_weights(cfg)
    prompt = synth.prompt(cfg, 40, stream=41)
    g = make_model(cfg, w)
    greedy = g.greedy(prompt, 30)
    g.close()
    m = make_model(cfg, w, draft_plan=[0, 3])
    rng = np.random.default_rng(9)
    out, acc = sv.selfspec_sampled(m, prompt, 30, 3, 1e-4,
                                   lambda c, k: rng.random(k) * 0.998 + 1e-3)
    m.check_error()
    assert out == greedy, (out[:10], greedy[:10])
    assert all(0 <= k <= 3 for k in acc)
    m.close()


def test_accept_sampled_argument_errors():
    torch = torch_cuda()
    import speculative_decoding_verify_pass_gb300 as sv
    m, cfg = _model(1000)
    tl = torch.zeros((17, 1000), dtype=torch.float32, device="cuda")
    u = torch.full((17,), 0.5, dtype=torch.float64, device="cuda")
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    for blk, dl, T in ((torch.zeros(17, dtype=torch.int32, device="cuda"), tl, 1.0),
                       (torch.zeros(3, dtype=torch.int32, device="cuda"), None, 1.0),
                       (torch.zeros(3, dtype=torch.int32, device="cuda"), tl, 0.0),
                       (torch.zeros(3, dtype=torch.int32, device="cuda"), tl, float("inf"))):
        with pytest.raises(sv.SpecError) as e:
            sv.spec_accept_sampled(m.h, tl, dl, blk, T, u, acc, tok)
        assert e.value.status == sv.SPEC_ERR_INVALID_ARG
    m.close()
