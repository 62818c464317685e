"""Sampled verification: the oracle of the rejection-sampling accept step.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline
leg of the benchmark are the only callers.

The LayerSkip summary (4.3.2, "Self-Verification") states the property only:
for sampling, rejection sampling makes the output distribution match the
full model's exactly, following the standard speculative decoding protocol.
The pages do not print the rule.  This module restates the standard rule of
speculative sampling (Leviathan, Kalman and Matias, "Fast Inference from
Transformers via Speculative Decoding", 2023; Chen et al., "Accelerating
Large Language Model Decoding with Speculative Sampling", 2023):

* p_j = softmax(target_logits[j] / T) is the target's distribution of the
  token after block[j]; q_j = softmax(draft_logits[j] / T) the draft's, from
  which block[j+1] was drawn.
* Draft j+1 is accepted when u_j < min(1, p_j(x) / q_j(x)), x = block[j+1],
  scanning j = 0, 1, ... until the first rejection.  Since u_j < 1 and
  q_j(x) > 0 for a token drawn from q_j, this is u_j * q_j(x) < p_j(x), and it
  is evaluated in the log domain from the logits,
  log u_j + log q_j(x) < log p_j(x) with log p_j(x) = (l_x - max l)/T -
  log(sum exp((l - max l)/T)), so that no probability underflows to zero.
* At the first rejection j, the next token is drawn from the residual
  norm(max(0, p_j - q_j)); if every draft is accepted, the bonus token is
  drawn from p_{n-1}.
* A draw from weights w with the uniform u is the smallest index i whose
  running sum w_0 + ... + w_i exceeds u * (w_0 + ... + w_{V-1}) (inverse CDF).

Everything is float64; the uniforms are inputs (u_accept for the n-1
drafts, then one u_final).
"""
from __future__ import annotations

import numpy as np


def softmax_t(logits, temperature: float) -> np.ndarray:
    """softmax(logits / T) in float64."""
    z = np.asarray(logits, dtype=np.float64) / float(temperature)
    e = np.exp(z - z.max())
    return e / e.sum()


def log_prob(logits, temperature: float, x: int) -> float:
    """log softmax(logits / T)[x] in float64, from the logits."""
    l = np.asarray(logits, dtype=np.float64)
    m = l.max()
    return (l[x] - m) / float(temperature) - np.log(np.sum(np.exp((l - m) / float(temperature))))


def accept_test(target_row, draft_row, temperature: float, x: int, u: float):
    """(accepted, margin): log u + log q(x) < log p(x), and the distance of
    the two sides."""
    lhs = np.log(u) + log_prob(draft_row, temperature, x)
    rhs = log_prob(target_row, temperature, x)
    return bool(lhs < rhs), abs(rhs - lhs)


def draw(weights, u: float) -> int:
    """Inverse-CDF draw: the smallest i with cumsum(weights)[i] > u * sum."""
    c = np.cumsum(np.asarray(weights, dtype=np.float64))
    i = int(np.searchsorted(c, u * c[-1], side="right"))
    return min(i, len(c) - 1)


def residual(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    """max(0, p - q); where p and q agree everywhere it is zero, and the
    residual draw falls back to p (the rejection then has probability 0)."""
    r = np.maximum(p - q, 0.0)
    return r if r.sum() > 0.0 else p


def accept_sampled(target_logits, draft_logits, block, temperature: float, u_accept, u_final: float):
    """(accept_len, next token) of one sampled verify pass of the n-token
    block [last accepted, x_1 .. x_{n-1}]: target_logits [n][V], draft_logits
    [n-1][V] (the draft's logits that produced x_1 .. x_{n-1})."""
    n = len(block)
    for j in range(n - 1):
        ok, _ = accept_test(target_logits[j], draft_logits[j], temperature, int(block[j + 1]), u_accept[j])
        if not ok:
            p = softmax_t(target_logits[j], temperature)
            q = softmax_t(draft_logits[j], temperature)
            return j, draw(residual(p, q), u_final)
    return n - 1, draw(softmax_t(target_logits[n - 1], temperature), u_final)


def decision_margins(target_logits, draft_logits, block, temperature: float, u_accept, u_final: float):
    """How far the oracle's decisions are from flipping: the smallest
    |log p(x) - log u - log q(x)| over the accept tests it made, and the
    distance of u_final * total from the nearest running-sum boundary of the
    draw, as a fraction of the total.  A GPU in fp32 may take the other
    branch only inside such a margin."""
    n = len(block)
    acc_margin = np.inf
    for j in range(n - 1):
        ok, mg = accept_test(target_logits[j], draft_logits[j], temperature, int(block[j + 1]), u_accept[j])
        acc_margin = min(acc_margin, mg)
        if not ok:
            w = residual(softmax_t(target_logits[j], temperature), softmax_t(draft_logits[j], temperature))
            break
    else:
        w = softmax_t(target_logits[n - 1], temperature)
    c = np.cumsum(w)
    t = u_final * c[-1]
    i = min(int(np.searchsorted(c, t, side="right")), len(c) - 1)
    lo = c[i - 1] if i > 0 else 0.0
    draw_margin = min(abs(t - lo), abs(c[i] - t)) / c[-1]
    return acc_margin, draw_margin
