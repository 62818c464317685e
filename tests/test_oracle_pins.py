"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself: each check is a closed form, a
special case that reduces to a library routine (numpy float64), an invariant
the pages state (greedy self-speculation is lossless; verifying n tokens
equals n decode steps; a rolled-back cache equals one that never held the
tail), brute force over small inputs, or a hand-worked table.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle
import synth
from conftest import small_gqa_cfg, small_moe_cfg

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_np(x):
    """Round float64/float32 values to bf16 (ties to even) with numpy bit ops."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def widen(bits):
    return synth.bf16_to_f32(bits).astype(np.float64)


# ----------------------------------------------------------------------------
# Layer plan and accept rule
# ----------------------------------------------------------------------------
def test_skip_sets_match_hand_worked_table():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "skip_sets.txt")) if l.strip() and l[0] != "#"]
    assert len(rows) >= 18
    for L, f, a, b in rows:
        L, f, a, b = int(L), float(f), int(a), int(b)
        keep = oracle.layer_skip_plan(L, f)
        skipped = [i for i in range(L) if i not in keep]
        assert skipped == list(range(a, b + 1)), (L, f)
        assert keep[0] == 0 and keep[-1] == L - 1       # first and last layers are always kept


@pytest.mark.parametrize("n", range(1, 17))
def test_accept_len_exhaustive(n):
    """All 2^(n-1) match patterns: accept_len is the index of the first mismatch
    (the longest matching prefix), n-1 when every draft matches."""
    for pattern in itertools.product([0, 1], repeat=n - 1):
        argmax_rows = list(range(100, 100 + n))
        block = [7] + [argmax_rows[j] if pattern[j] else argmax_rows[j] + 1 for j in range(n - 1)]
        first_miss = next((j for j, m in enumerate(pattern) if not m), n - 1)
        assert oracle.accept_len(block, argmax_rows) == first_miss


# ----------------------------------------------------------------------------
# Primitives
# ----------------------------------------------------------------------------
def test_bf16_round_ties_to_even():
    one = 1.0
    ulp = 2.0 ** -7                       # bf16 spacing just above 1
    assert oracle.bf16_round(one + ulp / 2) == one              # tie -> even (1.0)
    assert oracle.bf16_round(one + 1.5 * ulp) == one + 2 * ulp   # tie -> even
    assert oracle.bf16_round(one + ulp / 2 + 2 ** -20) == one + ulp
    assert oracle.bf16_round(-3.0) == -3.0


def test_gemm_matches_float64_matmul():
    rng = np.random.default_rng(0)
    W = synth.normal_bf16((37, 300), 9, 1)
    X = rng.standard_normal((5, 300)).astype(np.float32)
    Y = oracle.gemm(W, X)
    ref = X.astype(np.float64) @ widen(W).T
    # sequential fp32 sum: error <= K * eps32 * sum|terms|
    bound = 300 * 2 ** -24 * (np.abs(X).astype(np.float64) @ np.abs(widen(W)).T)
    assert np.all(np.abs(Y - ref) <= bound + 1e-30)
    assert Y.shape == (5, 37)


def test_rmsnorm_closed_forms():
    d, eps = 256, 1e-6
    g = synth.ones_bf16(d)
    h = oracle.rmsnorm(np.full(d, 3.0), g, eps)                 # constant c -> c/sqrt(c^2+eps)
    assert np.allclose(h, bf16_np(3.0 / math.sqrt(9.0 + eps)), rtol=0, atol=0)
    rng = np.random.default_rng(1)
    x = rng.standard_normal(d)
    h = oracle.rmsnorm(x, g, eps)
    ref = bf16_np(x / np.sqrt(np.mean(x * x) + eps))
    assert np.max(np.abs(h - ref)) <= 2 ** -7 * np.max(np.abs(ref))   # at most one bf16 step apart
    assert np.mean(h == ref) > 0.97
    g2 = synth.normal_bf16((d,), 3, 3, std=1.0)                  # gain multiplies elementwise
    h2 = oracle.rmsnorm(x, g2, eps)
    ref2 = bf16_np(x / np.sqrt(np.mean(x * x) + eps) * widen(g2))
    assert np.mean(h2 == ref2) > 0.97


def test_rope_closed_forms(tiny_oracle):
    hd = tiny_oracle.cfg.head_dim
    half = hd // 2
    rng = np.random.default_rng(2)
    v = rng.standard_normal(hd).astype(np.float32)
    assert np.array_equal(tiny_oracle.rope(v, 0), v)           # position 0 is the identity
    e0 = np.zeros(hd, dtype=np.float32)
    e0[0] = 1.0
    for pos in (1, 7, 100):
        r = tiny_oracle.rope(e0, pos)
        # pair (0, half) rotates by pos * theta^0 = pos radians: rotate-half pairing
        assert abs(r[0] - math.cos(pos)) < 1e-6 and abs(r[half] - math.sin(pos)) < 1e-6
        assert np.count_nonzero(np.abs(r) > 1e-7) == 2
    # last pair rotates by pos * theta^(-(hd-2)/hd)
    e_last = np.zeros(hd, dtype=np.float32)
    e_last[half - 1] = 1.0
    ang = 37 * tiny_oracle.cfg.rope_theta ** (-(hd - 2) / hd)
    r = tiny_oracle.rope(e_last, 37)
    assert abs(r[half - 1] - math.cos(ang)) < 1e-6 and abs(r[hd - 1] - math.sin(ang)) < 1e-6
    # rotation: norms kept, q(m).k(n) depends on m - n only
    q = rng.standard_normal(hd).astype(np.float32)
    k = rng.standard_normal(hd).astype(np.float32)
    assert abs(np.linalg.norm(tiny_oracle.rope(q, 55)) - np.linalg.norm(q)) < 1e-4
    d1 = float(np.dot(tiny_oracle.rope(q, 50), tiny_oracle.rope(k, 40)))
    d2 = float(np.dot(tiny_oracle.rope(q, 110), tiny_oracle.rope(k, 100)))
    assert abs(d1 - d2) < 1e-4


def test_attention_closed_forms():
    Hq, Hkv, hd = 8, 2, 64
    rng = np.random.default_rng(3)
    q = rng.standard_normal(Hq * hd).astype(np.float32)
    K = bf16_np(rng.standard_normal((1, Hkv * hd))).astype(np.float32)
    V = bf16_np(rng.standard_normal((1, Hkv * hd))).astype(np.float32)
    out = oracle.attend(q, K, V, Hq, Hkv, hd)                   # one key: softmax weight 1
    for h in range(Hq):
        assert np.array_equal(out[h * hd:(h + 1) * hd], V[0, (h // 4) * hd:(h // 4 + 1) * hd])
    nk = 9
    K = bf16_np(rng.standard_normal((nk, Hkv * hd))).astype(np.float32)
    V = bf16_np(rng.standard_normal((nk, Hkv * hd))).astype(np.float32)
    out = oracle.attend(np.zeros(Hq * hd, np.float32), K, V, Hq, Hkv, hd)   # q = 0: mean of values
    for h in range(Hq):
        ref = V[:, (h // 4) * hd:(h // 4 + 1) * hd].astype(np.float64).mean(0)
        assert np.max(np.abs(out[h * hd:(h + 1) * hd] - ref)) <= 2 ** -8 * np.max(np.abs(ref)) + 1e-6
    # query head h reads kv head h // (Hq/Hkv): constant values per kv head
    Vc = np.zeros((nk, Hkv * hd), np.float32)
    for j in range(Hkv):
        Vc[:, j * hd:(j + 1) * hd] = j + 1
    out = oracle.attend(q, K, Vc, Hq, Hkv, hd)
    for h in range(Hq):
        assert np.all(out[h * hd:(h + 1) * hd] == h // 4 + 1)
    # general case against float64 softmax
    out = oracle.attend(q, K, V, Hq, Hkv, hd)
    for h in range(Hq):
        kv = h // 4
        s = K[:, kv * hd:(kv + 1) * hd].astype(np.float64) @ q[h * hd:(h + 1) * hd] / math.sqrt(hd)
        p = np.exp(s - s.max())
        ref = p @ V[:, kv * hd:(kv + 1) * hd].astype(np.float64) / p.sum()
        assert np.max(np.abs(out[h * hd:(h + 1) * hd] - ref)) <= 2 ** -8 * np.max(np.abs(ref)) + 1e-6



# ----------------------------------------------------------------------------
# The fp64-accumulation build (same definition, long sums in fp64)
# ----------------------------------------------------------------------------
def test_acc64_gemm_is_the_correctly_rounded_dot_product():
    """bf16 x fp32 products are exact in fp64 and a 300-term fp64 sum is
    far inside half an fp32 ulp, so each output is float64 BLAS rounded to
    fp32 (a different result would mean a dropped or misplaced term)."""
    rng = np.random.default_rng(10)
    W = synth.normal_bf16((41, 300), 9, 2)
    X = bf16_np(rng.standard_normal((6, 300))).astype(np.float32)
    Y = oracle.gemm(W, X, acc64=True)
    ref = (X.astype(np.float64) @ widen(W).T).astype(np.float32)
    ulp = np.spacing(np.abs(ref))
    assert np.all(np.abs(Y.astype(np.float64) - ref) <= ulp)
    assert np.mean(Y == ref) > 0.99
    # and it is at least as close to float64 as the fp32 build
    y32 = oracle.gemm(W, X)
    exact = X.astype(np.float64) @ widen(W).T
    assert np.abs(Y - exact).sum() <= np.abs(y32 - exact).sum()


def test_acc64_rmsnorm_and_attention_against_float64():
    d, eps = 2560, 1e-6
    rng = np.random.default_rng(11)
    x = rng.standard_normal(d) * 3
    g = synth.normal_bf16((d,), 5, 3)
    h = oracle.rmsnorm(x, g, eps, acc64=True)
    x32 = x.astype(np.float32).astype(np.float64)
    rstd = np.float32(1.0 / np.sqrt(np.mean(x32 * x32) + eps))
    ref = bf16_np(x32.astype(np.float32) * rstd * widen(g).astype(np.float32))
    assert np.mean(h == ref) > 0.999
    assert np.max(np.abs(h - ref)) <= 2 ** -7 * np.max(np.abs(ref))
    Hq, Hkv, hd, nk = 4, 1, 128, 2048
    q = bf16_np(rng.standard_normal(Hq * hd)).astype(np.float32)
    K = bf16_np(rng.standard_normal((nk, Hkv * hd))).astype(np.float32)
    V = bf16_np(rng.standard_normal((nk, Hkv * hd))).astype(np.float32)
    out = oracle.attend(q, K, V, Hq, Hkv, hd, acc64=True)
    for hh in range(Hq):
        s = K.astype(np.float64) @ q[hh * hd:(hh + 1) * hd] / math.sqrt(hd)
        p = np.exp(s - s.max())
        ref = bf16_np(p @ V.astype(np.float64) / p.sum())
        got = out[hh * hd:(hh + 1) * hd]
        assert np.max(np.abs(got - ref)) <= 2 ** -8 * np.max(np.abs(ref)) + 1e-6
        assert np.mean(got == ref) > 0.95


def test_acc64_build_keeps_the_lossless_invariant(tiny_prompt):
    """Self-speculation equals greedy decoding in the fp64-accumulation build
    too (MLX self-speculation post), and the two builds agree on a shallow
    model to well inside the logit tolerance."""
    cfg = synth.tiny()
    w = synth.make_weights(cfg)
    o64 = oracle.Oracle(cfg, w, acc64=True)
    ref = oracle.greedy_generate(o64, tiny_prompt, 24)
    out, _ = oracle.selfspec_generate(o64, oracle.layer_skip_plan(cfg.n_layers, 0.3), tiny_prompt, 24, 4)
    assert out == ref
    o32 = oracle.Oracle(cfg, w)
    a, _, _ = o32.forward(o32.new_cache(), o32.full_plan, tiny_prompt, 0)
    b, _, _ = o64.forward(o64.new_cache(), o64.full_plan, tiny_prompt, 0)
    assert np.max(np.abs(a - b)) < 2e-2

def test_router_topk_against_sort():
    rng = np.random.default_rng(4)
    for trial in range(200):
        E, K = 64, 6
        lg = rng.standard_normal(E).astype(np.float32)
        if trial % 4 == 0:
            lg[rng.integers(0, E, 5)] = lg.max()               # exact ties at the top
        pr, ids, gates = oracle.route(lg, K)
        ref_p = np.exp(lg.astype(np.float64) - lg.max())
        ref_p /= ref_p.sum()
        assert abs(pr.sum() - 1.0) < 1e-5
        assert np.allclose(pr, ref_p, rtol=1e-5, atol=1e-7)
        order = sorted(range(E), key=lambda e: (-pr[e], e))     # larger first, lower id on ties
        assert list(ids) == order[:K]
        assert np.array_equal(gates, pr[ids])
    forced = np.array([5, 0, 63, 7, 9, 1], np.int32)
    pr, ids, gates = oracle.route(lg, 6, forced)
    assert list(ids) == list(forced) and np.array_equal(gates, pr[forced])


# ----------------------------------------------------------------------------
# Whole forward: first token at position 0 against a float64 library path
# ----------------------------------------------------------------------------
def _ref_first_token_logits(cfg, w, token):
    return _ref_first_token(cfg, w, token)[0]


def _ref_first_token(cfg, w, token):
    """At position 0 the rotation is the identity and each query sees one key,
    so attention returns v exactly; the rest is library float64 matmuls with
    the same bf16 rounding points.  Returns (logits, residual after each
    layer)."""
    d, eps = cfg.d_model, cfg.norm_eps
    xs = []
    x = widen(w.embed[token])

    def norm(v, g):
        return bf16_np(v / np.sqrt(np.mean(v * v) + eps) * widen(g))

    def ffn(h, wg, wu, wd):
        g = widen(wg) @ h
        u = widen(wu) @ h
        return widen(wd) @ bf16_np(g / (1 + np.exp(-g)) * u)

    for l, L in enumerate(w.layers):
        h = norm(x, L["attn_norm"])
        v = bf16_np(widen(L["wv"]) @ h)
        group = cfg.n_heads // cfg.n_kv_heads
        att = np.concatenate([v[(hh // group) * cfg.head_dim:(hh // group + 1) * cfg.head_dim]
                              for hh in range(cfg.n_heads)])
        x = x + widen(L["wo"]) @ att
        h = norm(x, L["ffn_norm"])
        if cfg.is_moe_layer(l):
            lg = widen(L["router"]) @ h
            p = np.exp(lg - lg.max())
            p /= p.sum()
            ids = sorted(range(cfg.n_experts), key=lambda e: (-p[e], e))[:cfg.top_k]
            y = sum(p[e] * ffn(h, L["e_gate"][e], L["e_up"][e], L["e_down"][e]) for e in ids)
            y = y + sum(ffn(h, L["s_gate"][s], L["s_up"][s], L["s_down"][s]) for s in range(cfg.n_shared_experts))
            x = x + y
        else:
            x = x + ffn(h, L["w_gate"], L["w_up"], L["w_down"])
        xs.append(x)
    return widen(w.lm_head_or_embed()) @ norm(x, w.final_norm), xs


@pytest.mark.parametrize("make", ["tiny", "gqa", "moe"])
def test_first_token_forward_matches_library_path(make):
    cfg = {"tiny": synth.tiny(), "gqa": small_gqa_cfg(), "moe": small_moe_cfg()}[make]
    w = synth.make_weights(cfg)
    orc = oracle.Oracle(cfg, w)
    for token in (0, 17, cfg.vocab - 1):
        cache = orc.new_cache()
        lg, _, _ = orc.forward(cache, orc.full_plan, [token], 0)
        ref = _ref_first_token_logits(cfg, w, token)
        err = np.abs(lg[0] - ref)
        # fp32 sums vs float64 sums may flip an occasional bf16 rounding of an
        # intermediate; a dropped term, sign error or transposed matrix moves
        # the logits by O(1) of their scale.
        scale = np.max(np.abs(ref))
        assert np.max(err) < 2e-2 * scale, (make, token, np.max(err), scale)
        assert np.mean(err) < 2e-3 * scale


def _rope64(v, pos, theta):
    """Rotate-half RoPE of head vectors v [..., hd] at `pos`, angles in float64."""
    hd = v.shape[-1]
    half = hd // 2
    ang = pos * theta ** (-2.0 * np.arange(half) / hd)
    c, s = np.cos(ang), np.sin(ang)
    a, b = v[..., :half], v[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def _ref_prompt_logits(cfg, w, tokens, rope_q=True, rope_k=True, causal=True):
    """Logits of every position of a prompt run from an empty cache, by
    float64 library matmuls with the oracle's bf16 rounding points: q and k
    rotated at their positions, then rounded; v rounded; query i attends to
    keys 0..i with softmax(q.k / sqrt(hd)); the attention output rounded.
    The switches plant wiring mistakes (RoPE left off q or k, attention over
    every key of the prompt) for the sensitivity checks."""
    d, eps, hd = cfg.d_model, cfg.norm_eps, cfg.head_dim
    T = len(tokens)
    group = cfg.n_heads // cfg.n_kv_heads
    X = np.stack([widen(w.embed[t]) for t in tokens])

    def norm(v, g):
        return bf16_np(v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps) * widen(g))

    def ffn(h, wg, wu, wd):
        g = h @ widen(wg).T
        u = h @ widen(wu).T
        return bf16_np(g / (1 + np.exp(-g)) * u) @ widen(wd).T

    for l, L in enumerate(w.layers):
        H = norm(X, L["attn_norm"])
        q = (H @ widen(L["wq"]).T).reshape(T, cfg.n_heads, hd)
        k = (H @ widen(L["wk"]).T).reshape(T, cfg.n_kv_heads, hd)
        v = bf16_np(H @ widen(L["wv"]).T).reshape(T, cfg.n_kv_heads, hd)
        for t in range(T):
            if rope_q:
                q[t] = _rope64(q[t], t, cfg.rope_theta)
            if rope_k:
                k[t] = _rope64(k[t], t, cfg.rope_theta)
        q, k = bf16_np(q), bf16_np(k)
        att = np.zeros((T, cfg.n_heads, hd))
        for t in range(T):
            keys = t + 1 if causal else T
            for hh in range(cfg.n_heads):
                kv = hh // group
                sc = k[:keys, kv] @ q[t, hh] / np.sqrt(hd)
                p = np.exp(sc - sc.max())
                att[t, hh] = bf16_np(p @ v[:keys, kv] / p.sum())
        X = X + att.reshape(T, -1) @ widen(L["wo"]).T
        H = norm(X, L["ffn_norm"])
        if cfg.is_moe_layer(l):
            Y = np.zeros_like(X)
            for t in range(T):
                lg = widen(L["router"]) @ H[t]
                p = np.exp(lg - lg.max())
                p /= p.sum()
                ids = sorted(range(cfg.n_experts), key=lambda e: (-p[e], e))[:cfg.top_k]
                Y[t] = sum(p[e] * ffn(H[t], L["e_gate"][e], L["e_up"][e], L["e_down"][e]) for e in ids)
                Y[t] += sum(ffn(H[t], L["s_gate"][s], L["s_up"][s], L["s_down"][s])
                            for s in range(cfg.n_shared_experts))
            X = X + Y
        else:
            X = X + ffn(H, L["w_gate"], L["w_up"], L["w_down"])
    return norm(X, w.final_norm) @ widen(w.lm_head_or_embed()).T


def _sharpened(cfg, w, factor=6.0):
    """The same weights with Wq and Wk scaled (then rounded to bf16) so that
    attention scores spread over several units: softmax is then far from
    uniform and which keys a query sees, and at which rotation, moves the
    output at the scale of the logits themselves."""
    import copy
    w2 = copy.copy(w)
    w2.layers = []
    for L in w.layers:
        L2 = dict(L)
        for key in ("wq", "wk"):
            f = np.asarray(bf16_np(widen(L[key]) * factor), dtype=np.float32)
            L2[key] = (f.view(np.uint32) >> 16).astype(np.uint16)
        w2.layers.append(L2)
    return w2


@pytest.mark.parametrize("make", ["tiny", "gqa", "moe"])
def test_prompt_forward_matches_library_path_at_later_positions(make):
    """Every position of a 6-token prompt (RoPE on q and k at positions
    1..5, causal multi-key grouped attention) against the float64 library
    path, with the same bounds as the position-0 pin.  The library path with
    RoPE left off q, off k, or with the causal mask dropped lands far outside
    those bounds, so each of those wiring mistakes in the oracle would fail
    here."""
    cfg = {"tiny": synth.tiny(), "gqa": small_gqa_cfg(), "moe": small_moe_cfg()}[make]
    w = _sharpened(cfg, synth.make_weights(cfg))
    orc = oracle.Oracle(cfg, w)
    toks = [int(t) for t in synth.prompt(cfg, 6, stream=31)]
    lg, _, _ = orc.forward(orc.new_cache(), orc.full_plan, toks, 0, logits_from=0)
    ref = _ref_prompt_logits(cfg, w, toks)
    scale = np.max(np.abs(ref))
    err = np.abs(lg - ref)
    assert np.max(err) < 2e-2 * scale and np.mean(err) < 2e-3 * scale, (make, np.max(err), np.mean(err), scale)
    for mutant in (dict(rope_q=False), dict(rope_k=False), dict(causal=False)):
        bad = _ref_prompt_logits(cfg, w, toks, **mutant)
        e = np.abs(bad - ref)[1:]          # position 0 is unaffected by all three
        assert np.mean(e) > 10 * 2e-3 * scale, (make, mutant, np.mean(e), scale)


@pytest.mark.parametrize("make", ["tiny", "gqa", "moe"])
def test_hidden_states_match_library_path(make):
    """The residual stream after every layer (the target hidden states the
    mlx-dflash README's draft conditions on), against the float64 library
    path at position 0."""
    cfg = {"tiny": synth.tiny(), "gqa": small_gqa_cfg(), "moe": small_moe_cfg()}[make]
    w = synth.make_weights(cfg)
    orc = oracle.Oracle(cfg, w)
    for token in (3, cfg.vocab - 2):
        hid = np.zeros((cfg.n_layers, 1, cfg.d_model), np.float32)
        orc.forward(orc.new_cache(), orc.full_plan, [token], 0, hidden=hid)
        _, xs = _ref_first_token(cfg, w, token)
        for l in range(cfg.n_layers):
            err = np.abs(hid[l, 0] - xs[l])
            scale = np.max(np.abs(xs[l]))
            assert np.max(err) < 2e-2 * scale and np.mean(err) < 2e-3 * scale, (make, token, l)


def test_hidden_state_taps_residual_identity_and_logits(tiny_prompt):
    """A layer whose O and down projections are zero leaves the residual
    stream unchanged, bit for bit; and the final norm and LM head applied to
    the last layer's hidden state give the oracle's logits."""
    import copy
    cfg = small_gqa_cfg()
    w = copy.deepcopy(synth.make_weights(cfg))
    L1 = w.layers[1]
    L1["wo"] = np.zeros_like(L1["wo"])
    L1["w_down"] = np.zeros_like(L1["w_down"])
    orc = oracle.Oracle(cfg, w)
    toks = [int(t) % cfg.vocab for t in tiny_prompt[:9]]
    hid = np.zeros((cfg.n_layers, len(toks), cfg.d_model), np.float32)
    lg, _, _ = orc.forward(orc.new_cache(), orc.full_plan, toks, 0, hidden=hid)
    assert np.array_equal(hid[1], hid[0])
    assert not np.array_equal(hid[2], hid[1])
    x = hid[-1].astype(np.float64)
    g = widen(w.final_norm)
    h = bf16_np(x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + cfg.norm_eps) * g)
    ref = h @ widen(w.lm_head_or_embed()).T
    assert np.max(np.abs(lg - ref)) < 1e-3 * np.max(np.abs(ref))
    assert [int(np.argmax(r)) for r in lg] == [int(np.argmax(r)) for r in ref]


# ----------------------------------------------------------------------------
# Invariants of the verify pass
# ----------------------------------------------------------------------------
def test_causality(tiny_oracle, tiny_prompt):
    orc = tiny_oracle
    c1, c2 = orc.new_cache(), orc.new_cache()
    toks = list(tiny_prompt[:20])
    a, _, _ = orc.forward(c1, orc.full_plan, toks, 0)
    toks2 = toks[:12] + [(t + 5) % orc.cfg.vocab for t in toks[12:]]
    b, _, _ = orc.forward(c2, orc.full_plan, toks2, 0)
    assert np.array_equal(a[:12], b[:12])
    assert not np.array_equal(a[12], b[12])


@pytest.mark.parametrize("cfgname", ["tiny", "gqa", "moe"])
def test_verify_block_equals_decode_steps(cfgname, tiny_oracle):
    """A verify pass over n tokens gives, row for row, the logits of n single-token
    decode steps (the LayerSkip summary, 4.3.2: verification is the same
    forward, run on all positions at once).  Bitwise in the oracle."""
    if cfgname == "tiny":
        orc = tiny_oracle
    else:
        cfg = small_gqa_cfg() if cfgname == "gqa" else small_moe_cfg()
        orc = oracle.Oracle(cfg, synth.make_weights(cfg))
    p = synth.prompt(orc.cfg, 40)
    ca, cb = orc.new_cache(), orc.new_cache()
    orc.forward(ca, orc.full_plan, p[:30], 0, logits_from=None)
    orc.forward(cb, orc.full_plan, p[:30], 0, logits_from=None)
    block = list(p[30:40])
    va, ida, _ = orc.forward(ca, orc.full_plan, block, 30, want_routing=True)
    for j, t in enumerate(block):
        vb, idb, _ = orc.forward(cb, orc.full_plan, [t], 30 + j, want_routing=True)
        assert np.array_equal(va[j], vb[0])
        if ida is not None:
            assert np.array_equal(ida[:, j], idb[:, 0])
    for s in range(orc.cfg.n_layers):
        assert np.array_equal(ca.read(s, 0, 40), cb.read(s, 0, 40))
        assert np.array_equal(ca.read(s, 1, 40), cb.read(s, 1, 40))


def test_rollback_equals_recompute(tiny_oracle, tiny_prompt):
    """Cropping a cache after a partial accept leaves the state of a cache that
    never held the rejected tail (the DFlash README crops the draft cache
    precisely on rejection)."""
    orc = tiny_oracle
    p = list(tiny_prompt)
    ca, cb = orc.new_cache(), orc.new_cache()
    orc.forward(ca, orc.full_plan, p[:50], 0, logits_from=None)
    orc.forward(ca, orc.full_plan, p[50:58], 50, logits_from=None)   # verify 8, accept 2 (+1)
    ca.truncate(53)
    orc.forward(cb, orc.full_plan, p[:53], 0, logits_from=None)
    la, _, _ = orc.forward(ca, orc.full_plan, [11, 12, 13], 53)
    lb, _, _ = orc.forward(cb, orc.full_plan, [11, 12, 13], 53)
    assert np.array_equal(la, lb)
    with pytest.raises(ValueError):
        ca.truncate(ca.len + 1)


@pytest.mark.parametrize("frac", [0.1, 0.2, 0.3, 0.4, 0.5])
@pytest.mark.parametrize("gamma", [1, 2, 3, 4, 5])
def test_selfspec_equals_greedy_tiny(tiny_oracle, tiny_prompt, frac, gamma):
    """Greedy self-speculation is lossless: same tokens as plain greedy, for
    every skip fraction and draft length (MLX self-speculation post)."""
    plan = oracle.layer_skip_plan(tiny_oracle.cfg.n_layers, frac)
    ref = _greedy_ref(tiny_oracle, tiny_prompt)
    out, acc = oracle.selfspec_generate(tiny_oracle, plan, tiny_prompt, 64, gamma)
    assert out == ref
    assert all(0 <= k <= gamma for k in acc)


_GREEDY = {}


def _greedy_ref(orc, prompt):
    key = (id(orc), len(prompt))
    if key not in _GREEDY:
        _GREEDY[key] = oracle.greedy_generate(orc, prompt, 64)
    return _GREEDY[key]


@pytest.mark.parametrize("gamma", [1, 3, 4, 7])
def test_selfspec_full_plan_accepts_everything(tiny_oracle, tiny_prompt, gamma):
    """A draft running every layer is the target itself: every draft is
    accepted (accept_len == gamma), which drives the bonus-token path."""
    out, acc = oracle.selfspec_generate(tiny_oracle, tiny_oracle.full_plan, tiny_prompt, 64, gamma)
    assert out == _greedy_ref(tiny_oracle, tiny_prompt)
    assert all(k == gamma for k in acc)


@pytest.mark.parametrize("alpha", [0.0, 0.5, 0.7, 0.9, 1.0])
def test_corrupted_drafts_accept_exactly_the_clean_prefix(tiny_oracle, tiny_prompt, alpha):
    """Drafts built from the true greedy continuation, each corrupted with
    probability 1 - alpha: the output stays greedy and accept_len equals the
    number of leading uncorrupted drafts, cycle by cycle."""
    ref = _greedy_ref(tiny_oracle, tiny_prompt)
    m = len(tiny_prompt)
    truth = list(tiny_prompt) + ref + [0] * 32
    expected = []
    counter = [0]

    def propose(seq, gamma):
        p = len(seq)
        clean = truth[p:p + gamma]
        d = synth.corrupt_drafts(np.array(clean), alpha, tiny_oracle.cfg.vocab, stream=counter[0])
        counter[0] += 1
        if p - m + gamma <= len(ref) - 1:
            expected.append(next((j for j in range(gamma) if d[j] != clean[j]), gamma))
        else:
            expected.append(None)
        return d

    out, acc = oracle.verify_with_drafts(tiny_oracle, tiny_prompt, 64, 5, propose)
    assert out == ref
    for e, k in zip(expected, acc):
        if e is not None:
            assert k == e
    if alpha == 1.0:
        assert all(k == 5 for k, e in zip(acc, expected) if e is not None)
    if alpha == 0.0:
        assert all(k == 0 for k in acc)


def test_tiny_greedy_golden(tiny_oracle, tiny_prompt):
    """Guards the oracle against drift: tokens written by
    tests/golden/make_golden.py (which calls only the oracle)."""
    path = os.path.join(GOLDEN, "tiny_greedy.txt")
    want = [int(t) for t in open(path).read().split("\n")[-2].split()]
    assert _greedy_ref(tiny_oracle, tiny_prompt) == want


def test_moe_per_token_routing_recorded():
    cfg = small_moe_cfg()
    orc = oracle.Oracle(cfg, synth.make_weights(cfg))
    c = orc.new_cache()
    p = synth.prompt(cfg, 12)
    lg, ids, gates = orc.forward(c, orc.full_plan, p, 0, want_routing=True)
    assert ids.shape == (cfg.n_layers, 12, cfg.top_k)
    assert np.all(ids[0] == -1)                     # layer 0 is dense
    assert np.all((ids[1:] >= 0) & (ids[1:] < cfg.n_experts))
    for l in range(1, cfg.n_layers):
        for t in range(12):
            assert len(set(ids[l, t])) == cfg.top_k
            assert np.all(np.diff(gates[l, t]) <= 0)   # ranked by probability
    # forcing the computed routing reproduces the logits bitwise
    c2 = orc.new_cache()
    probs = np.zeros((cfg.n_layers, 12, cfg.n_experts), np.float32)
    lg2, ids2, gates2 = orc.forward(c2, orc.full_plan, p, 0, want_routing=True, forced_ids=np.maximum(ids, 0),
                                    probs=probs)
    assert np.array_equal(lg, lg2)
    # the reported router probabilities: a distribution whose top-k (lowest id
    # first on ties) is the free choice, with the gates read off it
    assert np.all(probs[0] == 0)
    for l in range(1, cfg.n_layers):
        for t in range(12):
            pr = probs[l, t].astype(np.float64)
            assert abs(pr.sum() - 1.0) < 1e-5 and np.all(pr > 0)
            top = sorted(range(cfg.n_experts), key=lambda e: (-pr[e], e))[:cfg.top_k]
            assert list(ids[l, t]) == top
            assert np.array_equal(gates2[l, t], probs[l, t][ids[l, t]])


# ----------------------------------------------------------------------------
# Block-draft conditioning (mlx-dflash README, "Architecture")
# ----------------------------------------------------------------------------
def _identity_bits(d):
    eye = np.zeros((d, d), np.uint16)
    eye[np.arange(d), np.arange(d)] = 0x3F80          # bf16 1.0
    return eye


def test_context_append_of_embeddings_reproduces_layer0_kv():
    """With fc the identity and the taps holding token embeddings (exact in
    bf16), the features are the embeddings themselves and layer 0's appended
    keys and values are, bit for bit, those a forward of the same tokens
    writes: the appended path is layer 0's k/v path."""
    cfg = small_gqa_cfg()
    w = synth.make_weights(cfg)
    orc = oracle.Oracle(cfg, w)
    toks = synth.prompt(cfg, 11, stream=4)
    taps = np.zeros((1, 16, cfg.d_model), np.float32)
    taps[0, :11] = widen(w.embed[toks])
    ca = orc.new_cache()
    feat = orc.context_append(ca, _identity_bits(cfg.d_model), taps, 11)
    assert np.array_equal(feat, taps[0, :11]) and ca.len == 11
    cb = orc.new_cache()
    orc.forward(cb, orc.full_plan, toks, 0, logits_from=None)
    for which in (0, 1):
        assert np.array_equal(ca.read(0, which, 11), cb.read(0, which, 11))
    assert not np.array_equal(ca.read(1, 0, 11), cb.read(1, 0, 11))   # layer 1 saw other inputs


def test_context_append_fc_and_position_continuity():
    """fc against a float64 library matmul of the bf16-rounded concatenation;
    appending 5 rows then 6 equals appending the 11 at once, bit for bit (each
    row is independent and positions continue from the cache length)."""
    cfg = small_gqa_cfg()
    w = synth.make_weights(cfg)
    orc = oracle.Oracle(cfg, w)
    d, n_in = cfg.d_model, 3
    fc = synth.normal_bf16((d, n_in * d), 21, 1)
    rng = np.random.default_rng(7)
    taps = rng.standard_normal((n_in, 16, d)).astype(np.float32)
    c1 = orc.new_cache()
    feat = orc.context_append(c1, fc, taps, 11)
    concat = np.concatenate([bf16_np(taps[t, :11].astype(np.float64)) for t in range(n_in)], axis=1)
    ref = concat @ widen(fc).T
    assert np.max(np.abs(feat - ref)) < 1e-5 * np.max(np.abs(ref))
    c2 = orc.new_cache()
    first = taps.copy()
    orc.context_append(c2, fc, first, 5)
    second = np.zeros_like(taps)
    second[:, :6] = taps[:, 5:11]
    orc.context_append(c2, fc, second, 6)
    assert c2.len == 11
    for l in range(cfg.n_layers):
        for which in (0, 1):
            assert np.array_equal(c1.read(l, which, 11), c2.read(l, which, 11))
