"""Pins of the sampled-verification oracle (oracle/sampling.py).

The property the LayerSkip summary states (4.3.2, "Self-Verification"):
rejection sampling makes the output distribution match the full model's
exactly.  Checked here by Monte Carlo over the accept rule itself, with
planted mistakes that the same check must reject; plus the limits the rule
reduces to: a vanishing temperature gives the greedy accept of the DFlash
README ("Architecture", Accept), a draft equal to the target accepts every
draft, and the inverse-CDF draw on hand-worked weights."""
import numpy as np
import pytest

import oracle
from oracle import sampling as smp


def _emitted(tl, dl, x, u_acc, u_fin, T=1.0):
    """Tokens a pass emits: the accepted drafts, then the pass's own token."""
    k, tok = smp.accept_sampled(tl, dl, x, T, u_acc, u_fin)
    return list(x[1:k + 1]) + [tok]


def _mc_first_two(V, n, trials, seed, rule=None):
    """Monte Carlo of one pass over a block of n-1 drafts drawn from the
    draft's distributions: counts of the first emitted token, and of the
    second one among passes that emitted at least two."""
    rng = np.random.default_rng(seed)
    tl = rng.normal(size=(n, V)) * 1.5
    dl = tl[:n - 1] + rng.normal(size=(n - 1, V)) * 1.2       # a different draft distribution
    p = [smp.softmax_t(r, 1.0) for r in tl]
    q = [smp.softmax_t(r, 1.0) for r in dl]
    first = np.zeros(V)
    second = np.zeros(V)
    for _ in range(trials):
        x = [0] + [smp.draw(q[j], rng.random()) for j in range(n - 1)]
        u = rng.random(n)
        out = (rule or _emitted)(tl, dl, x, u[:n - 1], u[n - 1])
        first[out[0]] += 1
        if len(out) > 1:
            second[out[1]] += 1
    return p, first, second


def _within(counts, probs, sigmas=4.5):
    tot = counts.sum()
    dev = np.abs(counts - tot * probs)
    return bool(np.all(dev <= sigmas * np.sqrt(tot * probs * (1 - probs)) + 1e-9))


@pytest.mark.parametrize("n", [2, 3])
def test_emitted_tokens_follow_the_target_distribution(n):
    p, first, second = _mc_first_two(V=6, n=n, trials=60000, seed=11 + n)
    assert _within(first, p[0])
    assert second.sum() > 5000 and _within(second, p[1])


def test_planted_mistakes_change_the_distribution():
    """The Monte Carlo check has teeth: a residual drawn from p instead of
    max(0, p - q), and an accept test with the ratio inverted, both move the
    first token's distribution far outside the bound."""
    def wrong_residual(tl, dl, x, ua, uf):
        k, tok = smp.accept_sampled(tl, dl, x, 1.0, ua, uf)
        if k < len(x) - 1:
            tok = smp.draw(smp.softmax_t(tl[k], 1.0), uf)
        return list(x[1:k + 1]) + [tok]

    def inverted_ratio(tl, dl, x, ua, uf):
        p, q = smp.softmax_t(tl[0], 1.0), smp.softmax_t(dl[0], 1.0)   # accept when u < q/p: the wrong way round
        xx = x[1]
        if ua[0] < min(1.0, q[xx] / p[xx]):
            return [xx, smp.draw(smp.softmax_t(tl[1], 1.0), uf)]
        return [smp.draw(smp.residual(p, q), uf)]

    for rule in (wrong_residual, inverted_ratio):
        p, first, _ = _mc_first_two(V=6, n=2, trials=60000, seed=5, rule=rule)
        assert not _within(first, p[0], sigmas=8.0), rule.__name__


def test_vanishing_temperature_is_the_greedy_accept():
    rng = np.random.default_rng(3)
    V, n = 50, 6
    for trial in range(200):
        tl = rng.normal(size=(n, V))
        dl = rng.normal(size=(n - 1, V))
        a = [int(np.argmax(r)) for r in tl]
        # drafts: the target's own argmax for a random prefix, then anything;
        # each is the draft distribution's own argmax (what a draw from q is
        # as the temperature vanishes)
        k_true = int(rng.integers(0, n))
        x = [int(rng.integers(0, V))] + [a[j] if j < k_true else (a[j] + 1 + int(rng.integers(0, V - 1))) % V
                                         for j in range(n - 1)]
        for j in range(n - 1):
            dl[j, x[j + 1]] = dl[j].max() + 0.5
        k, tok = smp.accept_sampled(tl, dl, x, 1e-4, rng.random(n - 1) * 0.998 + 1e-3, float(rng.random()))
        assert k == oracle.accept_len(x, a), trial
        assert tok == a[k], trial


def test_draft_equal_to_target_accepts_every_draft():
    rng = np.random.default_rng(4)
    tl = rng.normal(size=(5, 30))
    x = [1, 2, 3, 4, 5]
    k, tok = smp.accept_sampled(tl, tl[:4], x, 0.8, [0.999999] * 4, 0.37)
    assert k == 4 and tok == smp.draw(smp.softmax_t(tl[4], 0.8), 0.37)


def test_inverse_cdf_draw_hand_worked():
    w = [1.0, 0.0, 3.0]
    assert smp.draw(w, 0.0) == 0
    assert smp.draw(w, 0.2) == 0          # 0.8 < 1
    assert smp.draw(w, 0.3) == 2          # 1.2: skips the zero weight
    assert smp.draw(w, 0.999999) == 2
    assert smp.draw([0.25, 0.25, 0.25, 0.25], 0.5) == 2
