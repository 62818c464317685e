"""Step-time model of speculative decoding used by the benchmark's predictions.

From "Speculative Decoding for Mixture-of-Experts Models: Expert Bytes,
Kernel Bandwidth and the Best Draft Length" (abstract): a step takes the
bytes each kernel requests over that kernel's effective bandwidth, plus fixed
time; with geometric acceptance the expected tokens of one verify of gamma
drafts is 1 + alpha + ... + alpha^gamma, the best draft length maximises
tokens per cycle time, and deduplicated expert reads win exactly when their
share of the per-slot bytes is below their bandwidth ratio.
"""
from __future__ import annotations

import math


def pass_bytes(cfg, n: int, ctx: int, plan=None) -> int:
    """Algorithmic bytes of one dense pass of n tokens at context ctx:
    weights of the executed layers, LM head, KV read over ctx, KV rows
    written, embedding rows."""
    layers = cfg.n_layers if plan is None else len(plan)
    d, hd = cfg.d_model, cfg.head_dim
    q_width, kv_width = cfg.n_heads * hd, cfg.n_kv_heads * hd
    weights = ((q_width + 2 * kv_width) * d + d * q_width + 3 * cfg.ffn_dim * d) * 2
    kv_row = 2 * kv_width * 2
    return layers * (weights + kv_row * (ctx + n)) + cfg.vocab * d * 2 + n * d * 2


def expert_bytes(cfg) -> int:
    """Bytes of one routed expert (gate, up, down)."""
    return 3 * cfg.expert_ffn * cfg.d_model * 2


def tokens_per_verify(alpha: float, gamma: int) -> float:
    """E[accepted drafts + 1] when P(accept >= j) = alpha^j, j <= gamma."""
    total, term = 0.0, 1.0
    for _ in range(gamma + 1):
        total += term
        term *= alpha
    return total


def mean_accept_truncated(alpha: float, max_len: int) -> float:
    """E[accept_len] = sum_{j=1..max_len} alpha^j."""
    return tokens_per_verify(alpha, max_len) - 1.0


def alpha_for_mean_accept(mean: float, max_len: int) -> float:
    """The alpha whose truncated-geometric accept length has the given mean."""
    lo, hi = 0.0, 1.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if mean_accept_truncated(mid, max_len) < mean:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def union_size_expected(n: int, n_experts: int, top_k: int, p_keep: float = 0.5) -> float:
    """E|experts used by n tokens| for traces where each token keeps the
    previous token's k experts with probability p_keep, else draws a fresh
    uniform k-subset: an expert is missed with probability
    (1 - k/E) * (p_keep + (1 - p_keep)(1 - k/E))^(n-1)."""
    miss_first = 1.0 - top_k / n_experts
    miss_next = p_keep + (1.0 - p_keep) * miss_first
    return n_experts * (1.0 - miss_first * miss_next ** (n - 1))


def union_size(ids_rows) -> int:
    """Distinct experts among the given rows of expert ids."""
    seen = set()
    for row in ids_rows:
        seen.update(int(e) for e in row)
    return len(seen)


def dedup_wins(byte_share: float, bandwidth_ratio: float) -> bool:
    """Deduplicated reads are faster iff bytes_dd/bytes_ps < B_dd/B_ps."""
    return byte_share < bandwidth_ratio


def first_win(pass_sizes, byte_shares, bandwidth_ratios):
    """Smallest pass size at which deduplication is faster, else None."""
    for n, u, r in zip(pass_sizes, byte_shares, bandwidth_ratios):
        if dedup_wins(u, r):
            return n
    return None


def best_gamma(alpha: float, verify_time, draft_time: float, gammas) -> int:
    """argmax_gamma tokens_per_verify(alpha, gamma) / (verify_time(gamma+1)
    + gamma*draft_time); ties go to the smaller gamma."""
    best, best_rate = None, -math.inf
    for g in gammas:
        rate = tokens_per_verify(alpha, g) / (verify_time(g + 1) + g * draft_time)
        if best is None or rate > best_rate * (1.0 + 1e-12):
            best, best_rate = g, rate
    return best


def fit_bandwidth(bytes_per_run, seconds_per_run):
    """Effective bandwidth of one operation from repeated isolated runs of the
    same bytes: the mean rate, and its relative spread (half the range of the
    per-run rates over their mean), used as the bandwidth error."""
    rates = [b / t for b, t in zip(bytes_per_run, seconds_per_run)]
    mean = sum(rates) / len(rates)
    return mean, (max(rates) - min(rates)) / (2.0 * mean)


def dedup_saving(bytes_ps, bytes_dd, bw_ps: float, bw_dd: float, err_ps: float, err_dd: float):
    """Time deduplication saves over per-slot reads on a pass whose expert
    operations request bytes_ps[l] / bytes_dd[l] per layer l, at bandwidths
    bw_ps / bw_dd with relative errors err_ps / err_dd.  A relative bandwidth
    error e moves a time b/B by at most b/B * e/(1-e); the bound adds both
    modes' moves.  Returns (saving, bound)."""
    t_ps = sum(bytes_ps) / bw_ps
    t_dd = sum(bytes_dd) / bw_dd
    bound = t_ps * err_ps / (1.0 - err_ps) + t_dd * err_dd / (1.0 - err_dd)
    return t_ps - t_dd, bound


def predicted_verify_times(t_plain: float, expert_time, pass_sizes):
    """Verify time per pass size from a plain one-token step's measured time
    and the predicted expert time per pass size (bytes over fitted
    bandwidth): the non-expert part is taken as the plain step's time less its
    own predicted expert time, and held fixed."""
    rest = t_plain - expert_time(1)
    return {n: rest + expert_time(n) for n in pass_sizes}


def gamma_staircase(alphas, verify_time, draft_time: float, gammas):
    """Best draft length for each acceptance rate."""
    return [best_gamma(float(a), verify_time, draft_time, gammas) for a in alphas]


def fit_time_model(byte_counts, seconds):
    """Least-squares fit of an operation's time as fixed time plus bytes over
    effective bandwidth, t = t0 + bytes / B, over runs of different byte
    counts.  Returns (t0, B, rel_err) with rel_err the largest relative
    residual |t - t0 - bytes/B| / t of the runs, used as the model's error."""
    n = len(byte_counts)
    mb = sum(byte_counts) / n
    mt = sum(seconds) / n
    sxx = sum((b - mb) ** 2 for b in byte_counts)
    sxy = sum((b - mb) * (t - mt) for b, t in zip(byte_counts, seconds))
    slope = sxy / sxx
    t0 = mt - slope * mb
    err = max(abs(t - t0 - slope * b) / t for b, t in zip(byte_counts, seconds))
    return t0, 1.0 / slope, err


def model_time(t0: float, bandwidth: float, byte_counts) -> float:
    """Summed time of operations of the given byte counts under the fit."""
    return sum(t0 + b / bandwidth for b in byte_counts)
