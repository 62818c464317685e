"""Seeded synthetic inputs for the verify pass (weights, prompts, drafts, routing, KV).

This module is shared by the CUDA path and the CPU oracle and holds no model
arithmetic: it only draws numbers.  Every value is a pure function of
(seed, stream, index) through a counter-based SplitMix64 generator
(``synth.c``), so both sides see the same bits.

Workload presets follow the five model shapes the speculative-decoding pages
work with (a tiny dense decoder, Qwen3-4B, Llama-3.1-8B, Qwen3-8B with a
16-token block draft as in the DFlash README, and a DeepSeek-V2-Lite-shaped MoE
as on the MoE speculative-decoding page); the weights are random-init
N(0, 0.02) bf16 because no trained checkpoint is used.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field, asdict

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "_synth.so")
_lib = None

# Seeds of the five input families (weights use WEIGHT_SEED_BASE + config index).
WEIGHT_SEED_BASE = 1234
PROMPT_SEED = 1
DRAFT_SEED = 2
ROUTING_SEED = 3
KV_SEED = 4

WEIGHT_STD = 0.02

# Tensor kinds in the stream id.
K_WQ, K_WK, K_WV, K_WO, K_GATE, K_UP, K_DOWN, K_ROUTER, K_SGATE, K_SUP, K_SDOWN = range(1, 12)
S_EMBED = 1
S_LMHEAD = 2


def build(force: bool = False) -> str:
    """Compile synth.c into _synth.so next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i64, i32, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        vp = ctypes.c_void_p
        lib.sv_key.restype = u64
        lib.sv_key.argtypes = [u64, u64]
        lib.sv_word.restype = u64
        lib.sv_word.argtypes = [u64, u64]
        lib.sv_uniform.restype = dbl
        lib.sv_uniform.argtypes = [u64, u64, u64]
        lib.sv_normal_bf16.argtypes = [vp, i64, u64, u64, i64, dbl]
        lib.sv_normal_f32.argtypes = [vp, i64, u64, u64, i64, dbl]
        lib.sv_const_bf16.argtypes = [vp, i64, ctypes.c_float]
        lib.sv_uniform_int.argtypes = [vp, i64, u64, u64, i32, i32]
        lib.sv_uniform_f64.argtypes = [vp, i64, u64, u64]
        _lib = lib
    return _lib


# ----------------------------------------------------------------------------
# Model shapes
# ----------------------------------------------------------------------------
@dataclass
class ModelConfig:
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int            # dense FFN width (layer 0 of the MoE model too)
    vocab: int
    rope_theta: float = 1e4
    norm_eps: float = 1e-6
    tied_embeddings: bool = False
    n_experts: int = 0      # 0: dense model
    top_k: int = 0
    expert_ffn: int = 0
    n_shared_experts: int = 0
    first_moe_layer: int = 1
    max_ctx: int = 4096
    index: int = 0          # position in the preset list (weight seed offset)

    def is_moe_layer(self, layer: int) -> bool:
        return self.n_experts > 0 and layer >= self.first_moe_layer

    @property
    def weight_seed(self) -> int:
        return WEIGHT_SEED_BASE + self.index

    def as_dict(self):
        return asdict(self)


def tiny(max_ctx: int = 512) -> ModelConfig:
    return ModelConfig("tiny", 4, 256, 4, 4, 64, 1024, 1024, rope_theta=1e4, max_ctx=max_ctx, index=0)


def qwen3_4b(max_ctx: int = 4096) -> ModelConfig:
    return ModelConfig("qwen3-4b", 36, 2560, 32, 8, 128, 9728, 151936, rope_theta=1e4,
                       tied_embeddings=True, max_ctx=max_ctx, index=1)


def llama31_8b(max_ctx: int = 4352) -> ModelConfig:
    return ModelConfig("llama-3.1-8b", 32, 4096, 32, 8, 128, 14336, 128256, rope_theta=5e5,
                       max_ctx=max_ctx, index=2)


def qwen3_8b(max_ctx: int = 4352) -> ModelConfig:
    return ModelConfig("qwen3-8b", 36, 4096, 32, 8, 128, 12288, 151936, rope_theta=1e4,
                       max_ctx=max_ctx, index=3)


def moe_v2lite(max_ctx: int = 2304) -> ModelConfig:
    return ModelConfig("moe-v2-lite", 27, 2048, 16, 16, 128, 10944, 102400, rope_theta=1e4,
                       n_experts=64, top_k=6, expert_ffn=1408, n_shared_experts=2,
                       first_moe_layer=1, max_ctx=max_ctx, index=4)


PRESETS = {"tiny": tiny, "qwen3-4b": qwen3_4b, "llama-3.1-8b": llama31_8b,
           "qwen3-8b": qwen3_8b, "moe-v2-lite": moe_v2lite}


def scaled(cfg: ModelConfig, **over) -> ModelConfig:
    """A copy of ``cfg`` with some fields replaced (smaller parity shapes)."""
    d = cfg.as_dict()
    d.update(over)
    return ModelConfig(**d)


# ----------------------------------------------------------------------------
# Weights
# ----------------------------------------------------------------------------
def stream_id(layer: int, kind: int, expert: int = -1) -> int:
    """Stream of one weight tensor: layer, kind and expert packed in 64 bits."""
    return ((layer + 1) << 24) | (kind << 16) | (expert + 1)


def normal_bf16(shape, seed: int, stream: int, std: float = WEIGHT_STD, first: int = 0) -> np.ndarray:
    """bf16 bits (uint16) of std * N(0,1), element i = stream index first + i."""
    out = np.empty(int(np.prod(shape)), dtype=np.uint16)
    _load().sv_normal_bf16(out.ctypes.data, out.size, seed, stream, first, std)
    return out.reshape(shape)


def normal_f32(shape, seed: int, stream: int, std: float = 1.0) -> np.ndarray:
    out = np.empty(int(np.prod(shape)), dtype=np.float32)
    _load().sv_normal_f32(out.ctypes.data, out.size, seed, stream, 0, std)
    return out.reshape(shape)


def ones_bf16(n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    _load().sv_const_bf16(out.ctypes.data, n, 1.0)
    return out


@dataclass
class Weights:
    """Host bf16 (uint16 bits) tensors in the usual row-major [out][in] form."""
    cfg: ModelConfig
    embed: np.ndarray = None
    lm_head: np.ndarray = None          # None when tied to embed
    final_norm: np.ndarray = None
    layers: list = field(default_factory=list)   # dict per layer

    def lm_head_or_embed(self):
        return self.embed if self.lm_head is None else self.lm_head


def make_weights(cfg: ModelConfig, seed: int | None = None) -> Weights:
    """All weights of ``cfg``: matrices N(0, 0.02) bf16, RMSNorm gains 1."""
    s = cfg.weight_seed if seed is None else seed
    d, hd = cfg.d_model, cfg.head_dim
    w = Weights(cfg)
    w.embed = normal_bf16((cfg.vocab, d), s, S_EMBED)
    w.lm_head = None if cfg.tied_embeddings else normal_bf16((cfg.vocab, d), s, S_LMHEAD)
    w.final_norm = ones_bf16(d)
    for l in range(cfg.n_layers):
        L = {
            "attn_norm": ones_bf16(d),
            "ffn_norm": ones_bf16(d),
            "wq": normal_bf16((cfg.n_heads * hd, d), s, stream_id(l, K_WQ)),
            "wk": normal_bf16((cfg.n_kv_heads * hd, d), s, stream_id(l, K_WK)),
            "wv": normal_bf16((cfg.n_kv_heads * hd, d), s, stream_id(l, K_WV)),
            "wo": normal_bf16((d, cfg.n_heads * hd), s, stream_id(l, K_WO)),
        }
        if cfg.is_moe_layer(l):
            fe = cfg.expert_ffn
            L["router"] = normal_bf16((cfg.n_experts, d), s, stream_id(l, K_ROUTER))
            L["e_gate"] = [normal_bf16((fe, d), s, stream_id(l, K_GATE, e)) for e in range(cfg.n_experts)]
            L["e_up"] = [normal_bf16((fe, d), s, stream_id(l, K_UP, e)) for e in range(cfg.n_experts)]
            L["e_down"] = [normal_bf16((d, fe), s, stream_id(l, K_DOWN, e)) for e in range(cfg.n_experts)]
            L["s_gate"] = [normal_bf16((fe, d), s, stream_id(l, K_SGATE, e)) for e in range(cfg.n_shared_experts)]
            L["s_up"] = [normal_bf16((fe, d), s, stream_id(l, K_SUP, e)) for e in range(cfg.n_shared_experts)]
            L["s_down"] = [normal_bf16((d, fe), s, stream_id(l, K_SDOWN, e)) for e in range(cfg.n_shared_experts)]
        else:
            f = cfg.ffn_dim
            L["w_gate"] = normal_bf16((f, d), s, stream_id(l, K_GATE))
            L["w_up"] = normal_bf16((f, d), s, stream_id(l, K_UP))
            L["w_down"] = normal_bf16((d, f), s, stream_id(l, K_DOWN))
        w.layers.append(L)
    return w


# ----------------------------------------------------------------------------
# Token streams
# ----------------------------------------------------------------------------
def uniform_ints(count: int, lo: int, hi: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(count, dtype=np.int32)
    _load().sv_uniform_int(out.ctypes.data, count, seed, stream, lo, hi)
    return out


def uniform_f64(count: int, seed: int, stream: int) -> np.ndarray:
    out = np.empty(count, dtype=np.float64)
    _load().sv_uniform_f64(out.ctypes.data, count, seed, stream)
    return out


def prompt(cfg: ModelConfig, length: int, seed: int = PROMPT_SEED, stream: int = 0) -> np.ndarray:
    """``length`` uniform token ids in [0, vocab)."""
    return uniform_ints(length, 0, cfg.vocab, seed, 0x70000 + stream)


def corrupt_drafts(true_tokens: np.ndarray, alpha: float, vocab: int, seed: int = DRAFT_SEED,
                   stream: int = 0) -> np.ndarray:
    """Draft tokens that equal ``true_tokens[j]`` with probability alpha and
    otherwise a uniform token different from it.  Fed to a greedy verifier
    whose argmax is ``true_tokens``, P(accept_len >= j) = alpha**j."""
    n = len(true_tokens)
    u = uniform_f64(n, seed, 0x80000 + 2 * stream)
    r = uniform_ints(n, 0, vocab - 1, seed, 0x80001 + 2 * stream)
    out = np.array(true_tokens, dtype=np.int32).copy()
    for j in range(n):
        if not (u[j] < alpha):
            t = int(r[j])
            out[j] = t + 1 if t >= int(true_tokens[j]) else t
    return out


def geometric_accept_lengths(count: int, alpha: float, max_len: int, seed: int = DRAFT_SEED,
                             stream: int = 0) -> np.ndarray:
    """accept_len draws with P(len >= j) = alpha**j, truncated at max_len."""
    u = uniform_f64(count * max_len, seed, 0x90000 + stream).reshape(count, max_len)
    acc = (u < alpha)
    out = np.zeros(count, dtype=np.int32)
    for i in range(count):
        k = 0
        while k < max_len and acc[i, k]:
            k += 1
        out[i] = k
    return out


def routing_trace(n_layers_moe: int, n_tokens: int, n_experts: int, top_k: int, p_reuse: float = 0.5,
                  seed: int = ROUTING_SEED, stream: int = 0) -> np.ndarray:
    """Expert ids [layer][token][k]: token 0 draws k distinct experts uniformly;
    each later token keeps the previous token's set with probability p_reuse,
    otherwise draws a fresh set.  Within a set, ids are in draw order."""
    out = np.zeros((n_layers_moe, n_tokens, top_k), dtype=np.int32)
    for l in range(n_layers_moe):
        st = 0xA0000 + (stream << 12) + l
        coin = uniform_f64(n_tokens, seed, st)
        draws = uniform_f64(n_tokens * n_experts, seed, st + 0x100000).reshape(n_tokens, n_experts)
        for t in range(n_tokens):
            if t > 0 and coin[t] < p_reuse:
                out[l, t] = out[l, t - 1]
                continue
            pool = list(range(n_experts))
            for j in range(top_k):
                idx = int(draws[t, j] * len(pool))
                idx = min(idx, len(pool) - 1)
                out[l, t, j] = pool.pop(idx)
    return out


def synthetic_kv(cfg: ModelConfig, layer: int, ctx: int, which: int, seed: int = KV_SEED) -> np.ndarray:
    """bf16 bits of N(0,1) keys (which=0) or values (which=1): [ctx][Hkv][hd]."""
    return normal_bf16((ctx, cfg.n_kv_heads, cfg.head_dim), seed, ((layer + 1) << 8) | which, std=1.0)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bits (uint16) to float32 values."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
