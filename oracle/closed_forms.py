"""Closed forms of the speculative-decoding step-time model (oracle side).

TEST INFRASTRUCTURE ONLY (tests and the benchmark's CPU/prediction legs).

Sources:

* MoE speculative-decoding page (abstract): a step's time is the bytes each
  kernel requests over that kernel's effective bandwidth plus fixed time;
  a deduplicating engine reads each selected expert once per pass, a per-slot
  engine once per (token, slot); deduplication is faster exactly where its
  share u(n) of the per-slot bytes is below its bandwidth ratio r(n); under
  geometric acceptance the best draft length is a monotone staircase in the
  acceptance rate.
* Geometric acceptance (the same page): P(accept_len >= j) = alpha**j, so the
  expected tokens emitted by one verify of gamma drafts is
  sum_{j=0..gamma} alpha**j (the accepted drafts plus the verifier's token).
* Synthetic routing traces: token 0 draws k of E experts; each later token
  keeps the previous set with probability 1/2 or draws afresh.  An expert is
  outside the union of n tokens' sets with probability
  (1 - k/E) * (1/2 + 1/2 (1 - k/E))**(n-1).

Byte counts are the algorithmic bytes of one pass: every weight byte of the
executed layers once, the LM head once, the KV cache read over the context,
the KV rows written for the block and the block's embedding rows.
"""
from __future__ import annotations

from dataclasses import dataclass

BF16 = 2


def expected_tokens(alpha: float, gamma: int) -> float:
    """E[tokens emitted per verify] = sum_{j=0}^{gamma} alpha^j."""
    return sum(alpha ** j for j in range(gamma + 1))


def expected_union(n: int, n_experts: int, top_k: int, p_reuse: float = 0.5) -> float:
    """E|U(n)| of the synthetic routing trace (fresh draws are uniform k-subsets)."""
    q = 1.0 - top_k / n_experts
    return n_experts * (1.0 - q * (p_reuse + (1.0 - p_reuse) * q) ** (n - 1))


@dataclass
class PassBytes:
    """Algorithmic bytes of one pass, split by kernel family."""
    qkv: int = 0
    o: int = 0
    ffn_dense: int = 0
    router: int = 0
    experts: int = 0            # unique experts (what a dedup engine requests)
    experts_per_slot: int = 0   # n * top_k expert reads (what a per-slot engine requests)
    shared: int = 0
    lm_head: int = 0
    kv_read: int = 0
    kv_write: int = 0
    embed: int = 0

    @property
    def total(self) -> int:
        return (self.qkv + self.o + self.ffn_dense + self.router + self.experts + self.shared +
                self.lm_head + self.kv_read + self.kv_write + self.embed)

    @property
    def total_per_slot(self) -> int:
        return self.total - self.experts + self.experts_per_slot


def pass_bytes(cfg, n: int, ctx: int, plan=None, unique_experts_per_layer=None) -> PassBytes:
    """Bytes of one pass of n tokens at context ctx over ``plan`` (default all layers).

    ``unique_experts_per_layer``: |U| per executed MoE layer (list or number);
    default min(E, n*k) is NOT assumed -- the caller passes the routing's union."""
    plan = list(range(cfg.n_layers)) if plan is None else list(plan)
    d, hd = cfg.d_model, cfg.head_dim
    b = PassBytes()
    kvw = cfg.n_kv_heads * hd
    moe_i = 0
    for l in plan:
        b.qkv += (cfg.n_heads * hd + 2 * kvw) * d * BF16
        b.o += d * cfg.n_heads * hd * BF16
        b.kv_read += 2 * kvw * ctx * BF16
        b.kv_write += 2 * kvw * n * BF16
        if cfg.n_experts > 0 and l >= cfg.first_moe_layer:
            per_expert = 3 * cfg.expert_ffn * d * BF16
            b.router += cfg.n_experts * d * BF16
            if unique_experts_per_layer is None:
                u = min(cfg.n_experts, n * cfg.top_k)
            elif isinstance(unique_experts_per_layer, (int, float)):
                u = unique_experts_per_layer
            else:
                u = unique_experts_per_layer[moe_i]
            b.experts += int(round(u * per_expert))
            b.experts_per_slot += n * cfg.top_k * per_expert
            b.shared += cfg.n_shared_experts * per_expert
            moe_i += 1
        else:
            b.ffn_dense += 3 * cfg.ffn_dim * d * BF16
    b.lm_head = cfg.vocab * d * BF16
    b.embed = n * d * BF16
    return b


def step_time(bytes_by_kernel: dict, bandwidth_by_kernel: dict, t_fixed: float = 0.0) -> float:
    """T = sum_k bytes_k / B_k + t_fixed."""
    return sum(bytes_by_kernel[k] / bandwidth_by_kernel[k] for k in bytes_by_kernel) + t_fixed


def dedup_faster(u_share: float, r_ratio: float) -> bool:
    """Deduplication wins exactly when u(n) < r(n)."""
    return u_share < r_ratio


def crossover(u_shares, r_ratios, pass_sizes):
    """First pass size at which deduplication is faster, or None."""
    for n, u, r in zip(pass_sizes, u_shares, r_ratios):
        if dedup_faster(u, r):
            return n
    return None


def speculation_wins(alpha: float, gamma: int, t_plain: float, t_verify: float, t_draft: float) -> bool:
    """Speculation beats plain decoding when the expected tokens per cycle,
    each worth one plain step, take longer plainly than one cycle:
    E[tau(gamma)] * T(1) > T_verify(gamma+1) + gamma * T_draft."""
    return expected_tokens(alpha, gamma) * t_plain > t_verify + gamma * t_draft


def best_draft_length(alpha: float, t_verify_of_n, t_draft: float, gammas) -> int:
    """gamma* = argmax_gamma E[tau(gamma)] / (T_verify(gamma+1) + gamma*T_draft);
    the smallest gamma wins ties."""
    best, best_rate = None, -1.0
    for g in gammas:
        rate = expected_tokens(alpha, g) / (t_verify_of_n(g + 1) + g * t_draft)
        if rate > best_rate * (1 + 1e-12):
            best, best_rate = g, rate
    return best
