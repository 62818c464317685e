"""Helpers of the `-m gpu` parity tests: model construction and comparisons.

Tolerances: logits within 2e-2 absolute + 2e-2 relative of the oracle
(bf16 weights and activations with fp32 accumulation on both sides; the two
differ in summation order and in where bf16 rounding happens).  Argmax
tokens, accept lengths and expert ids must match exactly, except where the
oracle's own margin between the two candidates is below 1e-3 (a near tie is
flagged, not failed)."""
import numpy as np
import pytest

ATOL = 2e-2
RTOL = 2e-2
TIE_GAP = 1e-3


def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def make_model(cfg, weights, draft_plan=None):
    import speculative_decoding_verify_pass_gb300 as sv
    return sv.Model(cfg, weights, draft_plan=draft_plan)


def assert_logits_close(gpu, ref, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), what + ": non-finite logits"
    err = np.abs(gpu - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), "%s: %d of %d logits outside tolerance (max err %.3g at ref %.3g)" % (
        what, bad.sum(), bad.size, err.max(), ref.flat[int(np.argmax(err))])


def argmax_mismatches(gpu_tokens, ref_logits):
    """Rows where the GPU argmax differs from the oracle's; raises unless the
    oracle's margin between the two tokens is a near tie.  Returns the
    flagged rows."""
    flagged = []
    for i, (g, row) in enumerate(zip(np.asarray(gpu_tokens).ravel(), np.asarray(ref_logits))):
        o = int(np.argmax(row))
        if int(g) != o:
            gap = float(row[o] - row[int(g)])
            assert gap < TIE_GAP, "row %d: GPU argmax %d vs oracle %d, oracle margin %.4g" % (i, g, o, gap)
            flagged.append(i)
    return flagged
