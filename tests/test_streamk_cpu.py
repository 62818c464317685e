"""The streaming GEMM's stream-K partition, restated on the host and checked
for every matrix of every workload shape, so that each reduction wait ends.

The kernel flattens a matrix's (tile, k-block) space, I = T * KBs stages
(128-row tiles, 64-wide k-blocks), and gives CTA c the contiguous range
[c*I/G, (c+1)*I/G) of G CTAs, G = min(I, SMs, 159*T).  A tile split between
CTAs is reduced by its first contributor (the CTA owning the tile's first
stage, ((i+1)*G - 1) / I); every other contributor stores one partial into
slot 2c (its range starts inside the tile) or 2c + 1 (otherwise) and adds
one arrival to the tile's counter; the reducer waits for contributors - 1
arrivals.  The checks: the ranges partition the space; the owner formula
names the CTA whose range holds each stage; each split tile has at most 160
contributors and is its reducer's last segment; and no two partials of one
launch share a slot.
"""
import pytest

import synth

ROWS, KB = 128, 64
MAX_CONTRIB = 160


def matrices(cfg):
    """(N, K) of every dense GEMM a pass of this shape runs."""
    d, hd = cfg.d_model, cfg.head_dim
    q, kv = cfg.n_heads * hd, cfg.n_kv_heads * hd
    out = [(q + 2 * kv, d), (d, q), (cfg.vocab, d)]
    if cfg.n_experts == 0 or cfg.first_moe_layer > 0:
        out += [(2 * cfg.ffn_dim, d), (d, cfg.ffn_dim)]
    if cfg.n_experts > 0:
        out += [(cfg.n_experts, d)]                       # router
    return out


def partition(N, K, sms):
    T, KBs = (N + ROWS - 1) // ROWS, K // KB
    I = T * KBs
    G = min(I, sms, 159 * T)
    return T, KBs, I, G


def owner(i, I, G):
    return ((i + 1) * G - 1) // I


def start(c, I, G):
    return c * I // G


SHAPES = [synth.tiny(), synth.qwen3_4b(), synth.llama31_8b(), synth.qwen3_8b(), synth.moe_v2lite(),
          synth.scaled(synth.qwen3_4b(), vocab=1000)]


@pytest.mark.parametrize("sms", [152, 148, 132, 7])
@pytest.mark.parametrize("cfg", SHAPES, ids=lambda c: c.name)
def test_streamk_partition_lets_every_reduction_finish(cfg, sms):
    for N, K in matrices(cfg):
        T, KBs, I, G = partition(N, K, sms)
        ranges = [(start(c, I, G), start(c + 1, I, G)) for c in range(G)]
        assert ranges[0][0] == 0 and ranges[-1][1] == I
        assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
        assert all(e > s for s, e in ranges)                       # no CTA without work
        for c, (s, e) in enumerate(ranges):
            assert owner(s, I, G) == c and owner(e - 1, I, G) == c
        slots = {}
        for t in range(T):
            cf, cl = owner(t * KBs, I, G), owner(t * KBs + KBs - 1, I, G)
            if cf == cl:
                continue                                           # whole tile in one CTA: no reduction
            assert cl - cf + 1 <= MAX_CONTRIB
            assert ranges[cf][1] <= (t + 1) * KBs                  # the tile is cf's last segment
            for c in range(cf + 1, cl + 1):
                slot = 2 * c + (0 if ranges[c][0] // KBs == t else 1)
                assert slot not in slots, (N, K, t, c, slots.get(slot))
                slots[slot] = (t, c)
