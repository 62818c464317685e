"""Python binding of the GB300 speculative-decoding verify-pass library.

Argument marshalling only: every function below forwards to the C ABI of
``include/spec.h`` (``libspecverify.so``, built for sm_103a by
``_build.build()``), passing device pointers of torch tensors and the current
torch CUDA stream.  All arithmetic of the verify pass runs in the library's
CUDA kernels; if the library is missing, importing the binding's functions
raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

SPEC_OK, SPEC_ERR_INVALID_ARG, SPEC_ERR_CAPACITY, SPEC_ERR_STATE, SPEC_ERR_CUDA, SPEC_ERR_TIMEOUT, SPEC_ERR_OOM = range(7)
SPEC_MOE_PER_SLOT, SPEC_MOE_DEDUP = 0, 1
SPEC_CACHE_TARGET, SPEC_CACHE_DRAFT = 0, 1
SPEC_MAX_BLOCK = 16

EXPORTED = ["spec_model_create", "spec_model_destroy", "spec_set_draft_plan", "spec_set_stream", "spec_prefill",
            "spec_draft_step", "spec_verify_step", "spec_kv_rollback", "spec_moe_mode", "spec_last_error",
            "spec_check_error", "spec_kv_len", "spec_kv_load", "spec_kv_export", "spec_kv_set_len",
            "spec_moe_force_routing", "spec_last_launch_count", "spec_profile_enable", "spec_profile_read",
            "spec_accept_from_logits_noalloc", "spec_trace_enable", "spec_trace_read", "spec_trace_kinds",
            "spec_set_taps", "spec_set_context_fc", "spec_context_append", "spec_batch_reserve",
            "spec_batch_kv_load", "spec_batch_kv_export", "spec_batch_set_len", "spec_batch_len",
            "spec_verify_batch", "spec_share_prefix", "spec_draft_step_logits", "spec_accept_sampled"]


class SpecError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("spec status %d: %s" % (status, msg))
        self.status = status


class ModelConfigC(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n_layers", "d_model", "n_heads", "n_kv_heads", "head_dim",
                                              "ffn_dim", "vocab")] + \
               [("rope_theta", ctypes.c_float), ("norm_eps", ctypes.c_float), ("tied_embeddings", ctypes.c_int32)] + \
               [(n, ctypes.c_int32) for n in ("n_experts", "top_k", "expert_ffn", "n_shared_experts",
                                              "first_moe_layer", "max_ctx")]


_VP = ctypes.c_void_p
_VPP = ctypes.POINTER(ctypes.c_void_p)


class LayerWeightsC(ctypes.Structure):
    _fields_ = [(n, _VP) for n in ("attn_norm", "ffn_norm", "wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down",
                                   "router")] + \
               [(n, _VPP) for n in ("e_gate", "e_up", "e_down", "s_gate", "s_up", "s_down")]


class WeightsC(ctypes.Structure):
    _fields_ = [("embed", _VP), ("lm_head", _VP), ("final_norm", _VP), ("layers", ctypes.POINTER(LayerWeightsC))]


_lib = None


def library():
    """Load libspecverify.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libspecverify.so is not built; run __graft_entry__.build() "
                           "(the CUDA path has no fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    i32, vp = ctypes.c_int32, ctypes.c_void_p
    sig = {
        "spec_model_create": [ctypes.POINTER(ModelConfigC), ctypes.POINTER(WeightsC), vp, i32, vp, ctypes.POINTER(vp)],
        "spec_model_destroy": [vp],
        "spec_set_draft_plan": [vp, vp, i32],
        "spec_set_stream": [vp, vp],
        "spec_prefill": [vp, vp, i32, vp],
        "spec_draft_step": [vp, vp, i32, vp],
        "spec_draft_step_logits": [vp, vp, i32, vp, vp],
        "spec_accept_sampled": [vp, vp, vp, vp, i32, ctypes.c_float, vp, vp, vp],
        "spec_verify_step": [vp, vp, i32, vp, vp, vp, vp, vp],
        "spec_kv_rollback": [vp, i32, i32],
        "spec_moe_mode": [vp, i32],
        "spec_set_taps": [vp, vp, i32, vp],
        "spec_set_context_fc": [vp, vp, i32],
        "spec_batch_reserve": [vp, i32],
        "spec_share_prefix": [vp, i32],
        "spec_batch_kv_load": [vp, i32, i32, vp, vp, i32],
        "spec_batch_kv_export": [vp, i32, i32, vp, vp, i32],
        "spec_batch_set_len": [vp, i32, i32],
        "spec_batch_len": [vp, i32, vp],
        "spec_verify_batch": [vp, vp, i32, i32, vp, vp, vp],
        "spec_context_append": [vp, vp, i32],
        "spec_check_error": [vp],
        "spec_kv_len": [vp, i32, ctypes.POINTER(i32)],
        "spec_kv_load": [vp, i32, i32, vp, vp, i32],
        "spec_kv_export": [vp, i32, i32, vp, vp, i32],
        "spec_kv_set_len": [vp, i32, i32],
        "spec_moe_force_routing": [vp, vp],
        "spec_last_launch_count": [vp],
        "spec_profile_enable": [vp, i32],
        "spec_profile_read": [vp, i32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double),
                              ctypes.POINTER(i32)],
        "spec_accept_from_logits_noalloc": [vp, i32, i32, vp, vp, vp, vp],
        "spec_trace_enable": [vp, i32],
        "spec_trace_read": [vp, vp, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)],
        "spec_trace_kinds": [vp, vp, i32, ctypes.POINTER(i32)],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = i32
    lib.spec_last_error.argtypes = []
    lib.spec_last_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status: int):
    if status != SPEC_OK:
        raise SpecError(status, library().spec_last_error().decode(errors="replace"))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


# ----------------------------------------------------------------------------
# Same-name wrappers of the C ABI (torch CUDA tensors in, status checked)
# ----------------------------------------------------------------------------
def spec_prefill(h, d_tokens, d_next_token):
    _check(library().spec_prefill(h, _ptr(d_tokens), int(d_tokens.numel()), _ptr(d_next_token)))


def spec_draft_step(h, d_tokens, d_draft_token):
    _check(library().spec_draft_step(h, _ptr(d_tokens), int(d_tokens.numel()), _ptr(d_draft_token)))


def spec_draft_step_logits(h, d_tokens, d_draft_token, d_logits=None):
    _check(library().spec_draft_step_logits(h, _ptr(d_tokens), int(d_tokens.numel()), _ptr(d_draft_token),
                                            _ptr(d_logits)))


def spec_verify_step(h, d_block, d_argmax, d_accept_len, d_logits=None, d_expert_ids=None, d_next_pair=None):
    _check(library().spec_verify_step(h, _ptr(d_block), int(d_block.numel()), _ptr(d_argmax), _ptr(d_accept_len),
                                      _ptr(d_logits), _ptr(d_expert_ids), _ptr(d_next_pair)))


def spec_accept_sampled(h, d_target_logits, d_draft_logits, d_block, temperature, d_uniforms, d_accept_len,
                        d_next_token):
    """Rejection-sampling accept: target logits [n][V], draft logits [n-1][V]
    (None for n == 1), block int32 [n], uniforms float64 [n]."""
    _check(library().spec_accept_sampled(h, _ptr(d_target_logits), _ptr(d_draft_logits), _ptr(d_block),
                                         int(d_block.numel()), float(temperature), _ptr(d_uniforms),
                                         _ptr(d_accept_len), _ptr(d_next_token)))


def spec_kv_rollback(h, which: int, new_len: int):
    _check(library().spec_kv_rollback(h, int(which), int(new_len)))


def spec_moe_mode(h, mode: int):
    _check(library().spec_moe_mode(h, int(mode)))


def spec_set_taps(h, layers, d_out=None):
    """Hidden-state taps: the residual stream after each of ``layers`` is
    written by every target verify pass to ``d_out`` [len(layers)][16][d_model]
    (fp32, device).  An empty list switches them off."""
    arr = (ctypes.c_int32 * max(len(layers), 1))(*[int(l) for l in layers])
    _check(library().spec_set_taps(h, arr if layers else None, len(layers), _ptr(d_out)))


def spec_set_context_fc(h, d_fc, n_in: int):
    _check(library().spec_set_context_fc(h, _ptr(d_fc), int(n_in)))


def spec_context_append(h, d_taps, m: int):
    _check(library().spec_context_append(h, _ptr(d_taps), int(m)))


def spec_share_prefix(h, enable: bool):
    _check(library().spec_share_prefix(h, 1 if enable else 0))


def spec_batch_reserve(h, nseq: int):
    _check(library().spec_batch_reserve(h, int(nseq)))


def spec_batch_kv_load(h, seq, slot, d_k, d_v, ctx):
    _check(library().spec_batch_kv_load(h, int(seq), int(slot), _ptr(d_k), _ptr(d_v), int(ctx)))


def spec_batch_kv_export(h, seq, slot, d_k, d_v, ctx):
    _check(library().spec_batch_kv_export(h, int(seq), int(slot), _ptr(d_k), _ptr(d_v), int(ctx)))


def spec_batch_set_len(h, seq: int, length: int):
    _check(library().spec_batch_set_len(h, int(seq), int(length)))


def spec_batch_len(h, seq: int) -> int:
    out = ctypes.c_int32(0)
    _check(library().spec_batch_len(h, int(seq), ctypes.byref(out)))
    return int(out.value)


def spec_verify_batch(h, d_blocks, d_argmax, d_accept, d_logits=None):
    """d_blocks: int32 device tensor [nseq][n]."""
    nseq, n = int(d_blocks.shape[0]), int(d_blocks.shape[1])
    _check(library().spec_verify_batch(h, _ptr(d_blocks), nseq, n, _ptr(d_argmax), _ptr(d_accept), _ptr(d_logits)))


def spec_check_error(h):
    _check(library().spec_check_error(h))


def spec_kv_len(h, which: int) -> int:
    out = ctypes.c_int32(0)
    _check(library().spec_kv_len(h, int(which), ctypes.byref(out)))
    return int(out.value)


def spec_kv_load(h, which, slot, d_k, d_v, ctx):
    _check(library().spec_kv_load(h, int(which), int(slot), _ptr(d_k), _ptr(d_v), int(ctx)))


def spec_kv_export(h, which, slot, d_k, d_v, ctx):
    _check(library().spec_kv_export(h, int(which), int(slot), _ptr(d_k), _ptr(d_v), int(ctx)))


def spec_kv_set_len(h, which, length):
    _check(library().spec_kv_set_len(h, int(which), int(length)))


def spec_moe_force_routing(h, d_ids):
    _check(library().spec_moe_force_routing(h, _ptr(d_ids)))


def spec_set_draft_plan(h, layers):
    arr = (ctypes.c_int32 * max(1, len(layers)))(*[int(x) for x in layers])
    _check(library().spec_set_draft_plan(h, arr if layers else None, len(layers)))


def spec_last_launch_count(h) -> int:
    return int(library().spec_last_launch_count(h))


def spec_profile_enable(h, enable: bool):
    _check(library().spec_profile_enable(h, int(bool(enable))))


EPI_QKV, EPI_RESID, EPI_SWIGLU, EPI_LMHEAD, EPI_ROUTER, EPI_EXPERT_SWIGLU, EPI_EXPERT_DOWN, EPI_STORE = range(8)
PROF_DENSE, PROF_ALL = -1, -2


def spec_profile_read(h, kind: int = PROF_DENSE):
    """(total ms, total bytes, launches) of the recorded launches of one kind."""
    ms, by, n = ctypes.c_double(0), ctypes.c_double(0), ctypes.c_int32(0)
    _check(library().spec_profile_read(h, int(kind), ctypes.byref(ms), ctypes.byref(by), ctypes.byref(n)))
    return float(ms.value), float(by.value), int(n.value)


def spec_trace_enable(h, enable: bool):
    _check(library().spec_trace_enable(h, int(bool(enable))))


def spec_trace_read(h, capacity: int = 512 * 1216 * 4):
    """Stamps of the last traced pass as an int64 array [ctas][phases][4]."""
    out = np.zeros(capacity, dtype=np.int64)
    nph, nct = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(library().spec_trace_read(h, ctypes.c_void_p(out.ctypes.data), capacity, ctypes.byref(nph),
                                     ctypes.byref(nct)))
    return out[:nct.value * nph.value * 4].reshape(nct.value, nph.value, 4)


def spec_trace_kinds(h, capacity: int = 4096):
    """Kind code of each phase or launch of the last traced pass."""
    out = np.zeros(capacity, dtype=np.int32)
    n = ctypes.c_int32(0)
    _check(library().spec_trace_kinds(h, ctypes.c_void_p(out.ctypes.data), capacity, ctypes.byref(n)))
    return out[:n.value].copy()


def spec_accept_from_logits_noalloc(d_logits, d_block, d_argmax, d_accept_len, stream=None):
    """Argmax rows and accept_len from caller-computed logits [n][vocab]; the
    library allocates nothing for this call (fixed in-library scratch).
    d_logits: contiguous float32 CUDA tensor [n][vocab]; d_block, d_argmax:
    int32 CUDA tensors of at least n entries; d_accept_len: int32, >= 1."""
    import torch
    if not (isinstance(d_logits, torch.Tensor) and d_logits.dim() == 2 and d_logits.dtype == torch.float32
            and d_logits.is_cuda and d_logits.is_contiguous()):
        raise SpecError(SPEC_ERR_INVALID_ARG, "d_logits must be a contiguous 2-D float32 CUDA tensor")
    n, vocab = int(d_logits.shape[0]), int(d_logits.shape[1])
    for name, t, need in (("d_block", d_block, n), ("d_argmax", d_argmax, n), ("d_accept_len", d_accept_len, 1)):
        if not (isinstance(t, torch.Tensor) and t.dtype == torch.int32 and t.is_cuda and t.is_contiguous()
                and t.numel() >= need):
            raise SpecError(SPEC_ERR_INVALID_ARG, "%s must be a contiguous int32 CUDA tensor of at least %d entries"
                            % (name, need))
    st = _stream() if stream is None else ctypes.c_void_p(stream)
    _check(library().spec_accept_from_logits_noalloc(_ptr(d_logits), n, vocab, _ptr(d_block), _ptr(d_argmax),
                                                     _ptr(d_accept_len), st))


# ----------------------------------------------------------------------------
# Model: uploads host bf16 weights, creates a handle, forwards calls
# ----------------------------------------------------------------------------
def _config_c(cfg) -> ModelConfigC:
    return ModelConfigC(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim, cfg.vocab,
                        float(cfg.rope_theta), float(cfg.norm_eps), int(bool(cfg.tied_embeddings)), cfg.n_experts,
                        cfg.top_k, cfg.expert_ffn, cfg.n_shared_experts, cfg.first_moe_layer, cfg.max_ctx)


class Model:
    """A library handle over host weights (uint16 bf16 bits, row-major).

    ``weights`` needs ``embed``, ``lm_head`` (or None when tied),
    ``final_norm`` and ``layers`` (one dict per layer with the keys used by
    ``synth.make_weights``).  The device copies made for creation are freed
    once the library has repacked them."""

    def __init__(self, cfg, weights, draft_plan=None, stream=None):
        import torch
        self.cfg = cfg
        self._torch = torch
        lib = library()
        keep = []

        def dev(a):
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to("cuda", non_blocking=False)
            keep.append(t)
            return ctypes.c_void_p(t.data_ptr())

        def dev_list(arrs):
            ptrs = (ctypes.c_void_p * len(arrs))(*[dev(a) for a in arrs])
            keep.append(ptrs)
            return ctypes.cast(ptrs, _VPP)

        layers = (LayerWeightsC * cfg.n_layers)()
        for l, L in enumerate(weights.layers):
            lw = layers[l]
            for key in ("attn_norm", "ffn_norm", "wq", "wk", "wv", "wo", "router"):
                if key in L:
                    setattr(lw, key, dev(L[key]))
            for key in ("w_gate", "w_up", "w_down"):
                if key in L:
                    setattr(lw, key, dev(L[key]))
            for key in ("e_gate", "e_up", "e_down", "s_gate", "s_up", "s_down"):
                if key in L and len(L[key]):
                    setattr(lw, key, dev_list(L[key]))
        wc = WeightsC(dev(weights.embed), dev(weights.lm_head) if weights.lm_head is not None else None,
                      dev(weights.final_norm), ctypes.cast(layers, ctypes.POINTER(LayerWeightsC)))
        plan = list(draft_plan or [])
        arr = (ctypes.c_int32 * max(1, len(plan)))(*plan)
        h = ctypes.c_void_p()
        cc = _config_c(cfg)
        st = ctypes.c_void_p(stream) if stream is not None else _stream()
        torch.cuda.synchronize()
        _check(lib.spec_model_create(ctypes.byref(cc), ctypes.byref(wc), arr if plan else None, len(plan), st,
                                     ctypes.byref(h)))
        self.h = h
        self.draft_plan = plan
        del keep
        torch.cuda.synchronize()

    def close(self):
        if getattr(self, "h", None):
            library().spec_model_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- thin forwards ------------------------------------------------------
    def _i32(self, n):
        return self._torch.zeros(n, dtype=self._torch.int32, device="cuda")

    def prefill(self, tokens):
        t = self._torch.as_tensor(tokens, dtype=self._torch.int32).to("cuda")
        nxt = self._i32(1)
        spec_prefill(self.h, t, nxt)
        return nxt

    def draft_step(self, d_tokens, out=None, logits=False):
        """Draft token of the last of d_tokens (1 or 2); with logits=True
        returns (token, logits [n][vocab])."""
        out = self._i32(1) if out is None else out
        if not logits:
            spec_draft_step(self.h, d_tokens, out)
            return out
        lg = self._torch.empty((d_tokens.numel(), self.cfg.vocab), dtype=self._torch.float32, device="cuda")
        spec_draft_step_logits(self.h, d_tokens, out, lg)
        return out, lg

    def verify(self, d_block, logits=False, expert_ids=False, next_pair=None):
        n = d_block.numel()
        am = self._i32(n)
        acc = self._i32(1)
        lg = self._torch.empty((n, self.cfg.vocab), dtype=self._torch.float32, device="cuda") if logits else None
        ids = None
        if expert_ids:
            ids = self._torch.empty((self.cfg.n_layers, n, self.cfg.top_k), dtype=self._torch.int32, device="cuda")
        spec_verify_step(self.h, d_block, am, acc, lg, ids, next_pair)
        return am, acc, lg, ids

    def rollback(self, which, new_len):
        spec_kv_rollback(self.h, which, new_len)

    def accept_sampled(self, target_logits, draft_logits, d_block, temperature, uniforms):
        """(accept_len, next token) device tensors of the rejection-sampling
        accept; uniforms: n float64 values (host or device)."""
        torch = self._torch
        u = torch.as_tensor(uniforms, dtype=torch.float64).to("cuda")
        acc = self._i32(1)
        tok = self._i32(1)
        spec_accept_sampled(self.h, target_logits, draft_logits, d_block, temperature, u, acc, tok)
        return acc, tok

    def kv_len(self, which):
        return spec_kv_len(self.h, which)

    def moe_mode(self, mode):
        spec_moe_mode(self.h, mode)

    def set_context_fc(self, fc_bits):
        """Block-draft conditioning: fc as bf16 bits [d_model][n_in*d_model]
        (host array); uploaded, then repacked by the library."""
        torch = self._torch
        n_in = fc_bits.shape[1] // self.cfg.d_model
        dev = torch.from_numpy(np.ascontiguousarray(fc_bits).view(np.int16)).to("cuda")
        spec_set_context_fc(self.h, dev, n_in)
        del dev

    def context_append(self, taps, m):
        """Append m context positions from tapped hidden states (a device
        fp32 tensor [n_in][16][d_model], e.g. a target's set_taps buffer)."""
        spec_context_append(self.h, taps, m)

    def share_prefix(self, enable=True):
        """The draft's leading layers use the target's KV cache (the draft
        cache is reallocated and emptied)."""
        spec_share_prefix(self.h, enable)

    def batch_reserve(self, nseq):
        spec_batch_reserve(self.h, nseq)

    def batch_kv_load(self, seq, slot, k_bits, v_bits):
        torch = self._torch
        k = torch.from_numpy(np.ascontiguousarray(k_bits).view(np.int16)).to("cuda")
        v = torch.from_numpy(np.ascontiguousarray(v_bits).view(np.int16)).to("cuda")
        spec_batch_kv_load(self.h, seq, slot, k, v, k_bits.shape[0])
        torch.cuda.synchronize()

    def batch_kv_export(self, seq, slot, ctx):
        c = self.cfg
        k = self._torch.empty((ctx, c.n_kv_heads, c.head_dim), dtype=self._torch.int16, device="cuda")
        v = self._torch.empty_like(k)
        spec_batch_kv_export(self.h, seq, slot, k, v, ctx)
        self._torch.cuda.synchronize()
        return k.cpu().numpy().view(np.uint16), v.cpu().numpy().view(np.uint16)

    def batch_set_len(self, seq, length):
        spec_batch_set_len(self.h, seq, length)

    def batch_len(self, seq):
        return spec_batch_len(self.h, seq)

    def verify_batch(self, d_blocks, logits=False):
        """d_blocks: int32 device tensor [nseq][n]; returns (argmax [nseq][n],
        accept [nseq], logits [nseq*n][V] or None)."""
        torch = self._torch
        nseq, n = d_blocks.shape
        am = torch.empty((nseq, n), dtype=torch.int32, device="cuda")
        acc = torch.empty(nseq, dtype=torch.int32, device="cuda")
        lg = torch.empty((nseq * n, self.cfg.vocab), dtype=torch.float32, device="cuda") if logits else None
        spec_verify_batch(self.h, d_blocks, am, acc, lg)
        return am, acc, lg

    def set_taps(self, layers):
        """Tap the residual stream after ``layers`` in every verify pass;
        returns the fp32 device buffer [len(layers)][16][d_model] the passes
        write (None when ``layers`` is empty)."""
        self._taps = None
        if layers:
            self._taps = self._torch.zeros((len(layers), 16, self.cfg.d_model), dtype=self._torch.float32, device="cuda")
        spec_set_taps(self.h, list(layers), self._taps)
        return self._taps

    def check_error(self):
        spec_check_error(self.h)

    def force_routing(self, ids):
        """ids: int array [n_layers][16][top_k] (or None to return to top-k)."""
        if ids is None:
            spec_moe_force_routing(self.h, None)
            return
        t = self._torch.as_tensor(np.ascontiguousarray(ids, dtype=np.int32)).to("cuda")
        spec_moe_force_routing(self.h, t)

    def set_draft_plan(self, layers):
        spec_set_draft_plan(self.h, layers)
        self.draft_plan = list(layers)

    def kv_load(self, which, slot, k_bits, v_bits):
        k = self._torch.from_numpy(np.ascontiguousarray(k_bits).view(np.int16)).to("cuda")
        v = self._torch.from_numpy(np.ascontiguousarray(v_bits).view(np.int16)).to("cuda")
        spec_kv_load(self.h, which, slot, k, v, k_bits.shape[0])
        self._torch.cuda.synchronize()

    def kv_export(self, which, slot, ctx):
        c = self.cfg
        k = self._torch.empty((ctx, c.n_kv_heads, c.head_dim), dtype=self._torch.int16, device="cuda")
        v = self._torch.empty_like(k)
        spec_kv_export(self.h, which, slot, k, v, ctx)
        self._torch.cuda.synchronize()
        return k.cpu().numpy().view(np.uint16), v.cpu().numpy().view(np.uint16)

    def kv_set_len(self, which, length):
        spec_kv_set_len(self.h, which, length)

    def launches(self):
        return spec_last_launch_count(self.h)

    # -- loops of C calls ---------------------------------------------------
    def greedy(self, prompt, max_new):
        """Plain greedy decoding through verify passes of one token."""
        torch = self._torch
        out = [int(self.prefill(prompt).item())]
        blk = self._i32(1)
        while len(out) < max_new:
            blk.fill_(out[-1])
            am, _, _, _ = self.verify(blk)
            out.append(int(am.item()))
        return out

    def selfspec(self, prompt, max_new, gamma):
        """Greedy self-speculative decoding: gamma draft steps over the kept
        layers, one verify pass of gamma+1 tokens, accept, roll back both
        caches.  Returns (tokens, accept lengths)."""
        torch = self._torch
        p = [int(t) for t in prompt]
        y = int(self.prefill(p).item())
        out = [y]
        seq = p + out
        accepts = []
        dlen = len(p)
        while len(out) < max_new:
            pos = len(seq) - 1
            feed = seq[dlen:pos + 1]
            drafts = []
            for _ in range(gamma):
                t = torch.tensor(feed, dtype=torch.int32, device="cuda")
                d = int(self.draft_step(t).item())
                dlen += len(feed)
                drafts.append(d)
                feed = [d]
            block = torch.tensor([seq[pos]] + drafts, dtype=torch.int32, device="cuda")
            am, acc, _, _ = self.verify(block)
            k = int(acc.item())
            a = am.cpu().tolist()
            accepts.append(k)
            emitted = drafts[:k] + [a[k]]
            out += emitted
            seq += emitted
            self.rollback(SPEC_CACHE_TARGET, pos + k + 1)
            dlen = min(pos + k + 1, dlen)
            self.rollback(SPEC_CACHE_DRAFT, dlen)
        return out[:max_new], accepts


def selfspec_sampled(model, prompt, max_new, gamma, temperature, uniforms):
    """Self-speculative decoding with sampling: the draft samples each
    proposal from its own distribution at `temperature`, the target verifies
    the block by rejection sampling (spec_accept_sampled), both caches are
    rolled back to the accepted length.  ``uniforms(cycle, count)`` returns the
    float64 uniforms a cycle draws (gamma draft draws, then gamma accept tests
    and the final draw).  The prompt's last token is the first block's head.
    Returns (tokens, accept lengths)."""
    import torch
    m = model
    p = [int(t) for t in prompt]
    one = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.prefill(p[:-1])
    seq = list(p)
    out, accepts = [], []
    dlen = len(p) - 1
    cycle = 0
    while len(out) < max_new:
        pos = len(seq) - 1
        u = list(uniforms(cycle, 2 * gamma + 1))
        feed = seq[dlen:pos + 1]
        drafts, dlog = [], []
        for i in range(gamma):
            t = torch.tensor(feed, dtype=torch.int32, device="cuda")
            _, lg = m.draft_step(t, logits=True)
            row = lg[-1:].contiguous()
            _, x = m.accept_sampled(row, None, one, temperature, [u[i]])
            d = int(x.item())
            dlen += len(feed)
            drafts.append(d)
            dlog.append(row)
            feed = [d]
        block = torch.tensor([seq[pos]] + drafts, dtype=torch.int32, device="cuda")
        _, _, tl, _ = m.verify(block, logits=True)
        dl = torch.cat(dlog, 0) if dlog else None
        k, tok = m.accept_sampled(tl, dl, block, temperature, u[gamma:])
        k = int(k.item())
        emitted = drafts[:k] + [int(tok.item())]
        accepts.append(k)
        out += emitted
        seq += emitted
        m.rollback(SPEC_CACHE_TARGET, pos + k + 1)
        dlen = min(pos + k + 1, dlen)
        m.rollback(SPEC_CACHE_DRAFT, dlen)
        cycle += 1
    return out[:max_new], accepts


def layer_skip_plan(n_layers: int, skip_frac: float):
    """Kept layers of the contiguous middle-skip draft (MLX self-speculation
    post, "Code -> the implementation"): drop max(1, round(n_layers*skip_frac))
    layers (round half to even) starting at (n_layers - dropped) // 2."""
    drop = max(1, int(round(n_layers * skip_frac)))
    first = (n_layers - drop) // 2
    return [l for l in range(n_layers) if l < first or l >= first + drop]


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)
