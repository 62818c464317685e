"""CPU oracle of the greedy speculative-decoding verify pass.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline
leg of the benchmark are the only callers.  Nothing here is shared with the
CUDA path except the seeded inputs of ``synth``.

``oracle.c`` holds the forward pass (fp32, sequential sums, bf16 rounding at
the declared points); this module holds the loops that the pages describe on
top of it:

* ``layer_skip_plan`` -- the contiguous middle-skip draft of the MLX
  self-speculation post ("Code -> the implementation": n_skip =
  max(1, round(L * f)), start = (L - n_skip) // 2, keep every other layer).
* ``accept_len`` -- the greedy cumulative-product match of the DFlash README
  ("Architecture", Accept step) and of the LayerSkip summary (4.3.2 step 3:
  keep the drafted tokens up to the first mismatch, then the verifier's own
  token).
* ``greedy_generate`` / ``selfspec_generate`` -- plain greedy decoding and the
  draft -> verify -> accept -> roll back loop; the MLX post and the DFlash
  README both state that the greedy self-speculative output must equal the
  plain greedy output, token for token.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIBS = {False: os.path.join(_HERE, "_oracle.so"), True: os.path.join(_HERE, "_oracle64.so")}
_lib = {}

(T_EMBED, T_LMHEAD, T_FINALNORM, T_ATTN_NORM, T_FFN_NORM, T_WQ, T_WK, T_WV, T_WO,
 T_GATE, T_UP, T_DOWN, T_ROUTER, T_EGATE, T_EUP, T_EDOWN, T_SGATE, T_SUP, T_SDOWN) = range(19)


class _Cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("n_layers", "d_model", "n_heads", "n_kv_heads", "head_dim",
                                             "ffn_dim", "vocab")] + \
               [("rope_theta", ctypes.c_float), ("norm_eps", ctypes.c_float)] + \
               [(n, ctypes.c_int) for n in ("n_experts", "top_k", "expert_ffn", "n_shared",
                                             "first_moe_layer", "max_ctx")]


def build(force: bool = False, acc64: bool = False) -> str:
    """Compile oracle.c (gcc, OpenMP, no FMA contraction so x86 and Arm agree).
    ``acc64`` selects the build whose long sums accumulate in fp64."""
    path = _LIBS[bool(acc64)]
    if force or not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
        tmp = path + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]
                              + (["-DORC_ACC64"] if acc64 else []) + ["-o", tmp, _SRC, "-lm"])
        os.replace(tmp, path)
    return path


def build_all(force: bool = False) -> None:
    """Both builds: fp32 accumulation (the oracle) and fp64 accumulation."""
    build(force, False)
    build(force, True)


def _load(acc64: bool = False):
    acc64 = bool(acc64)
    if acc64 not in _lib:
        lib = ctypes.CDLL(build(acc64=acc64))
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        lib.orc_create.restype = vp
        lib.orc_create.argtypes = [ctypes.POINTER(_Cfg)]
        lib.orc_destroy.argtypes = [vp]
        lib.orc_set.argtypes = [vp, i32, i32, i32, vp]
        lib.orc_set.restype = i32
        lib.orc_cache_create.restype = vp
        lib.orc_cache_create.argtypes = [vp, i32]
        lib.orc_cache_destroy.argtypes = [vp]
        lib.orc_cache_len.argtypes = [vp]
        lib.orc_cache_len.restype = i32
        lib.orc_cache_truncate.argtypes = [vp, i32]
        lib.orc_cache_truncate.restype = i32
        lib.orc_cache_load.argtypes = [vp, i32, i32, vp, vp]
        lib.orc_cache_load.restype = i32
        lib.orc_cache_set_len.argtypes = [vp, i32]
        lib.orc_cache_set_len.restype = i32
        lib.orc_cache_read.argtypes = [vp, i32, i32, i32, vp]
        lib.orc_cache_read.restype = i32
        lib.orc_forward.argtypes = [vp, vp, vp, i32, vp, i32, i32, vp, i32, vp, vp, vp, vp, vp]
        lib.orc_forward.restype = i32
        lib.orc_context_append.argtypes = [vp, vp, vp, i32, vp, i32, vp]
        lib.orc_context_append.restype = i32
        lib.orc_argmax.argtypes = [vp, i32]
        lib.orc_argmax.restype = i32
        lib.orc_bf16_round.argtypes = [ctypes.c_float]
        lib.orc_bf16_round.restype = ctypes.c_float
        lib.orc_set_threads.argtypes = [i32]
        lib.orc_get_threads.restype = i32
        lib.orc_gemm.argtypes = [vp, i32, i32, vp, i32, vp]
        lib.orc_rmsnorm.argtypes = [vp, vp, i32, ctypes.c_float, vp]
        lib.orc_rope.argtypes = [vp, vp, i32]
        lib.orc_attend.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp]
        lib.orc_route.argtypes = [vp, i32, i32, vp, vp, vp]
        _lib[acc64] = lib
    return _lib[acc64]


def set_threads(n: int) -> None:
    _load().orc_set_threads(int(n))


def get_threads() -> int:
    return int(_load().orc_get_threads())


def bf16_round(x: float) -> float:
    return float(_load().orc_bf16_round(float(x)))


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


# ----------------------------------------------------------------------------
# Primitives (the functions the forward is built from), exposed for the pins
# ----------------------------------------------------------------------------
def gemm(w_bits: np.ndarray, x: np.ndarray, acc64: bool = False) -> np.ndarray:
    """Y[i][r] = sum_k W[r][k] X[i][k], k in order, in the build's accumulator."""
    W = np.ascontiguousarray(w_bits, dtype=np.uint16)
    X = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    N, K = W.shape
    Y = np.empty((X.shape[0], N), dtype=np.float32)
    _load(acc64).orc_gemm(_ptr(W), N, K, _ptr(X), X.shape[0], _ptr(Y))
    return Y


def rmsnorm(x: np.ndarray, g_bits: np.ndarray, eps: float, acc64: bool = False) -> np.ndarray:
    """bf16(x * rsqrt(mean(x^2) + eps) * g)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    g = np.ascontiguousarray(g_bits, dtype=np.uint16)
    h = np.empty_like(x)
    _load(acc64).orc_rmsnorm(_ptr(x), _ptr(g), x.size, eps, _ptr(h))
    return h


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, n_heads: int, n_kv_heads: int, head_dim: int,
           acc64: bool = False):
    """One token's grouped-query attention over nk cached keys.
    q [Hq*hd]; K, V [nk][Hkv*hd]; returns bf16-rounded [Hq*hd]."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    K = np.ascontiguousarray(K, dtype=np.float32)
    V = np.ascontiguousarray(V, dtype=np.float32)
    out = np.empty(n_heads * head_dim, dtype=np.float32)
    _load(acc64).orc_attend(_ptr(q), _ptr(K), _ptr(V), K.shape[0], n_heads, n_kv_heads, head_dim, _ptr(out))
    return out


def route(logits: np.ndarray, top_k: int, forced=None):
    """(probabilities, ids, gates) of one token's router."""
    pr = np.ascontiguousarray(logits, dtype=np.float32).copy()
    ids = np.empty(top_k, dtype=np.int32)
    gates = np.empty(top_k, dtype=np.float32)
    f = None if forced is None else np.ascontiguousarray(forced, dtype=np.int32)
    _load().orc_route(_ptr(pr), pr.size, top_k, _ptr(f) if f is not None else None, _ptr(ids), _ptr(gates))
    return pr, ids, gates


class Cache:
    """Per-plan KV cache of the oracle (slot s holds layer plan[s])."""

    def __init__(self, model: "Oracle", n_slots: int):
        self._lib = model._lib
        self.n_slots = n_slots
        self.model = model
        self.h = self._lib.orc_cache_create(model.h, n_slots)

    def __del__(self):
        if getattr(self, "h", None):
            self._lib.orc_cache_destroy(self.h)
            self.h = None

    @property
    def len(self) -> int:
        return int(self._lib.orc_cache_len(self.h))

    def truncate(self, new_len: int) -> None:
        if self._lib.orc_cache_truncate(self.h, int(new_len)) != 0:
            raise ValueError("truncate to %d of a cache holding %d" % (new_len, self.len))

    def load(self, slot: int, k_bits: np.ndarray, v_bits: np.ndarray) -> None:
        k = np.ascontiguousarray(k_bits, dtype=np.uint16)
        v = np.ascontiguousarray(v_bits, dtype=np.uint16)
        ctx = k.shape[0]
        if self._lib.orc_cache_load(self.h, slot, ctx, _ptr(k), _ptr(v)) != 0:
            raise ValueError("bad cache load")

    def set_len(self, n: int) -> None:
        if self._lib.orc_cache_set_len(self.h, int(n)) != 0:
            raise ValueError("bad length")

    def read(self, slot: int, which: int, ctx: int) -> np.ndarray:
        c = self.model.cfg
        out = np.empty((ctx, c.n_kv_heads * c.head_dim), dtype=np.float32)
        if self._lib.orc_cache_read(self.h, slot, which, ctx, _ptr(out)) != 0:
            raise ValueError("bad cache read")
        return out


class Oracle:
    """The oracle model over host bf16 weights from ``synth.make_weights``."""

    def __init__(self, cfg, weights, acc64: bool = False):
        self._lib = _load(acc64)
        self.acc64 = bool(acc64)
        self.cfg = cfg
        self.weights = weights      # keeps the host buffers alive
        c = _Cfg(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim,
                 cfg.vocab, cfg.rope_theta, cfg.norm_eps, cfg.n_experts, cfg.top_k, cfg.expert_ffn,
                 cfg.n_shared_experts, cfg.first_moe_layer, cfg.max_ctx)
        self.h = self._lib.orc_create(ctypes.byref(c))
        self._keep = []
        self._set(T_EMBED, -1, -1, weights.embed)
        if weights.lm_head is not None:
            self._set(T_LMHEAD, -1, -1, weights.lm_head)
        self._set(T_FINALNORM, -1, -1, weights.final_norm)
        for l, L in enumerate(weights.layers):
            for kind, key in ((T_ATTN_NORM, "attn_norm"), (T_FFN_NORM, "ffn_norm"), (T_WQ, "wq"),
                              (T_WK, "wk"), (T_WV, "wv"), (T_WO, "wo"), (T_GATE, "w_gate"),
                              (T_UP, "w_up"), (T_DOWN, "w_down"), (T_ROUTER, "router")):
                if key in L:
                    self._set(kind, l, -1, L[key])
            for kind, key in ((T_EGATE, "e_gate"), (T_EUP, "e_up"), (T_EDOWN, "e_down"),
                              (T_SGATE, "s_gate"), (T_SUP, "s_up"), (T_SDOWN, "s_down")):
                for e, t in enumerate(L.get(key, [])):
                    self._set(kind, l, e, t)

    def _set(self, kind, layer, expert, arr):
        a = np.ascontiguousarray(arr, dtype=np.uint16)
        self._keep.append(a)
        if self._lib.orc_set(self.h, kind, layer, expert, _ptr(a)) != 0:
            raise ValueError("bad tensor registration")

    def __del__(self):
        if getattr(self, "h", None):
            self._lib.orc_destroy(self.h)
            self.h = None

    def rope(self, v: np.ndarray, pos: int) -> np.ndarray:
        """Rotate-half RoPE of one head vector at ``pos`` (float32 copy)."""
        out = np.ascontiguousarray(v, dtype=np.float32).copy()
        self._lib.orc_rope(self.h, _ptr(out), int(pos))
        return out

    @property
    def full_plan(self):
        return list(range(self.cfg.n_layers))

    def new_cache(self, n_slots: int | None = None) -> Cache:
        return Cache(self, self.cfg.n_layers if n_slots is None else n_slots)

    def forward(self, cache: Cache, plan, tokens, pos0: int, logits_from: int | None = 0,
                want_routing: bool = False, forced_ids=None, probs=None, hidden=None):
        """Run ``tokens`` at positions pos0.. through ``plan``; returns
        (logits[rows][V] or None, ids or None, gates or None).  ``probs``, a
        float32 array [len(plan)][n][n_experts], receives the router
        probabilities of the MoE layers; ``hidden``, a float32 array
        [len(plan)][n][d_model], the residual stream after each layer."""
        plan_a = np.ascontiguousarray(plan, dtype=np.int32)
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        n = len(tok)
        c = self.cfg
        logits = None
        if logits_from is not None and logits_from < n:
            logits = np.empty((n - logits_from, c.vocab), dtype=np.float32)
        ids = gates = None
        if want_routing and c.n_experts > 0:
            ids = np.full((len(plan_a), n, c.top_k), -1, dtype=np.int32)
            gates = np.zeros((len(plan_a), n, c.top_k), dtype=np.float32)
        forced = None
        if forced_ids is not None:
            forced = np.ascontiguousarray(forced_ids, dtype=np.int32)
            assert forced.shape == (len(plan_a), n, c.top_k)
        if probs is not None:
            assert probs.dtype == np.float32 and probs.flags.c_contiguous
            assert probs.shape == (len(plan_a), n, c.n_experts)
        if hidden is not None:
            assert hidden.dtype == np.float32 and hidden.flags.c_contiguous
            assert hidden.shape == (len(plan_a), n, c.d_model)
        rc = self._lib.orc_forward(self.h, cache.h, _ptr(plan_a), len(plan_a), _ptr(tok), n, int(pos0),
                                   _ptr(logits) if logits is not None else None,
                                   int(logits_from) if logits is not None else 0,
                                   _ptr(ids) if ids is not None else None,
                                   _ptr(gates) if gates is not None else None,
                                   _ptr(forced) if forced is not None else None,
                                   _ptr(probs) if probs is not None else None,
                                   _ptr(hidden) if hidden is not None else None)
        if rc != 0:
            raise ValueError("oracle forward rejected its arguments")
        return logits, ids, gates


    def context_append(self, cache: Cache, fc_bits: np.ndarray, taps: np.ndarray, rows: int) -> np.ndarray:
        """The block draft's conditioning (mlx-dflash README, "Architecture"):
        features = fc . bf16(concat of the taps of rows 0..rows-1), then every
        layer appends the keys and values of those positions computed from the
        features.  fc_bits: bf16 bits [d_model][n_in * d_model]; taps: float32
        [n_in][16][d_model].  Returns the features [rows][d_model]."""
        c = self.cfg
        fc = np.ascontiguousarray(fc_bits, dtype=np.uint16)
        tp = np.ascontiguousarray(taps, dtype=np.float32)
        n_in = tp.shape[0]
        assert tp.shape == (n_in, 16, c.d_model) and fc.shape == (c.d_model, n_in * c.d_model)
        feat = np.empty((rows, c.d_model), dtype=np.float32)
        if self._lib.orc_context_append(self.h, cache.h, _ptr(fc), n_in, _ptr(tp), int(rows), _ptr(feat)) != 0:
            raise ValueError("oracle context append rejected its arguments")
        return feat


# ----------------------------------------------------------------------------
# Loops over the forward
# ----------------------------------------------------------------------------
def argmax(row: np.ndarray) -> int:
    """Lowest index among the maxima (np.argmax keeps the first maximum)."""
    return int(np.argmax(row))


def layer_skip_plan(n_layers: int, skip_frac: float):
    """Kept layers of the middle-skip draft: n_skip = max(1, round(L*f)) layers
    starting at (L - n_skip) // 2 are dropped (Python round, half to even)."""
    n_skip = max(1, round(n_layers * skip_frac))
    start = (n_layers - n_skip) // 2
    skip = set(range(start, start + n_skip))
    return [i for i in range(n_layers) if i not in skip]


def accept_len(block, argmax_rows) -> int:
    """Greedy cumulative-product match: the number of leading j in
    [0, n-1) with block[j+1] == argmax_rows[j]."""
    k = 0
    match = 1
    for j in range(len(block) - 1):
        match *= int(int(block[j + 1]) == int(argmax_rows[j]))
        k += match
    return k


def greedy_generate(orc: Oracle, prompt, max_new: int, plan=None):
    """Plain greedy decoding: prefill, then one token per forward."""
    plan = orc.full_plan if plan is None else list(plan)
    cache = orc.new_cache(len(plan))
    logits, _, _ = orc.forward(cache, plan, prompt, 0, logits_from=len(prompt) - 1)
    out = [argmax(logits[-1])]
    while len(out) < max_new:
        logits, _, _ = orc.forward(cache, plan, [out[-1]], cache.len, logits_from=0)
        out.append(argmax(logits[-1]))
    return out


def selfspec_generate(orc: Oracle, draft_plan, prompt, max_new: int, gamma: int):
    """Greedy self-speculative decoding with a layer-subset draft.

    Each cycle: the draft (its own KV cache over ``draft_plan``) first catches
    up on the accepted tokens it has not seen, then proposes gamma tokens one
    at a time; the full model verifies [y, d1..d_gamma] in one pass; the
    accepted prefix plus the verifier's token at the first mismatch (or the
    bonus token after a full accept) are emitted; both caches are rolled back
    to the accepted length.  Returns (tokens, accept lengths per cycle)."""
    full = orc.full_plan
    tc = orc.new_cache(len(full))
    dc = orc.new_cache(len(draft_plan))
    prompt = [int(t) for t in prompt]
    logits, _, _ = orc.forward(tc, full, prompt, 0, logits_from=len(prompt) - 1)
    orc.forward(dc, draft_plan, prompt, 0, logits_from=None)
    out = [argmax(logits[-1])]
    seq = prompt + out
    accepts = []
    while len(out) < max_new:
        p = len(seq) - 1                   # position of y, the last accepted token
        feed = seq[dc.len:p + 1]
        drafts = []
        for _ in range(gamma):
            lg, _, _ = orc.forward(dc, draft_plan, feed, dc.len, logits_from=len(feed) - 1)
            drafts.append(argmax(lg[-1]))
            feed = [drafts[-1]]
        block = [seq[p]] + drafts
        lg, _, _ = orc.forward(tc, full, block, p, logits_from=0)
        a = [argmax(r) for r in lg]
        k = accept_len(block, a)
        accepts.append(k)
        emitted = drafts[:k] + [a[k]]
        out += emitted
        seq += emitted
        tc.truncate(p + k + 1)
        dc.truncate(min(p + k + 1, dc.len))
    return out[:max_new], accepts


def verify_with_drafts(orc: Oracle, prompt, max_new: int, gamma: int, propose):
    """The verify / accept / roll-back loop with drafts from ``propose(seq, gamma)``
    (any token source, e.g. seeded corruptions of the true continuation).
    Returns (tokens, accept lengths per cycle)."""
    full = orc.full_plan
    tc = orc.new_cache(len(full))
    prompt = [int(t) for t in prompt]
    logits, _, _ = orc.forward(tc, full, prompt, 0, logits_from=len(prompt) - 1)
    out = [argmax(logits[-1])]
    seq = prompt + out
    accepts = []
    while len(out) < max_new:
        p = len(seq) - 1
        drafts = [int(t) for t in propose(seq, gamma)]
        block = [seq[p]] + drafts
        lg, _, _ = orc.forward(tc, full, block, p, logits_from=0)
        a = [argmax(r) for r in lg]
        k = accept_len(block, a)
        accepts.append(k)
        emitted = drafts[:k] + [a[k]]
        out += emitted
        seq += emitted
        tc.truncate(p + k + 1)
    return out[:max_new], accepts
