"""Helpers of the `-m gpu` parity tests: model construction and comparisons.

Tolerances: logits within 2e-2 absolute + 2e-2 relative of the oracle
(bf16 weights and activations with fp32 accumulation on both sides; the two
differ in summation order and in where bf16 rounding happens).  Argmax
tokens, accept lengths and expert ids must match exactly, except where the
oracle's own margin between the two candidates is below 1e-3 (a near tie is
flagged, not failed).

At full depth and width that logit tolerance is beyond what fp32
accumulation itself reproduces: the fp32-accumulating oracle and its
fp64-accumulating build drift apart by more than it (tests/golden/
fullsize_floor.txt).  There the reference is the fp64 build, and the GPU's
deviation from it may be at most FLOOR_FACTOR times the fp32 oracle's own
deviation from it; where the floor is inside the tolerance, the tolerance
holds as stated."""
import numpy as np
import pytest

ATOL = 2e-2
RTOL = 2e-2
TIE_GAP = 1e-3
FLOOR_FACTOR = 1.5


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


def argmax_mismatches(gpu_tokens, ref_logits, tie_gap=TIE_GAP):
    """Rows where the GPU argmax differs from the oracle's; raises unless the
    oracle's margin between the two tokens is a near tie (below tie_gap).
    Returns the flagged rows."""
    flagged = []
    for i, (g, row) in enumerate(zip(np.asarray(gpu_tokens).ravel(), np.asarray(ref_logits))):
        o = int(np.argmax(row))
        if int(g) != o:
            gap = float(row[o] - row[int(g)])
            assert gap < tie_gap, "row %d: GPU argmax %d vs oracle %d, oracle margin %.4g" % (i, g, o, gap)
            flagged.append(i)
    return flagged


def load_floor():
    """Cases of tests/golden/fullsize_floor.txt: name -> dict(preset, layers,
    ctx, n, stream, mean, max, share, route_mismatch, route_dp); the last
    two are None for dense models."""
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "fullsize_floor.txt")
    out = {}
    for line in open(path):
        if not line.strip() or line[0] == "#":
            continue
        f = line.split()
        opt = [None if v == "-" else float(v) for v in f[9:11]]
        out[f[0]] = dict(preset=f[1], layers=int(f[2]), ctx=int(f[3]), n=int(f[4]), stream=int(f[5]),
                         mean=float(f[6]), max=float(f[7]), share=float(f[8]),
                         route_mismatch=opt[0], route_dp=opt[1])
    return out


def assert_within_floor(gpu, ref64, floor, what=""):
    """GPU logits against the fp64-accumulating oracle.  Where the fp32
    oracle itself stays inside ATOL + RTOL (floor share 0) every logit must;
    elsewhere the GPU's mean and max deviation and its share outside the
    tolerance may be at most FLOOR_FACTOR times the fp32 oracle's."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref64, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), what + ": non-finite logits"
    if floor["share"] == 0.0:
        assert_logits_close(gpu, ref, what)
        return
    err = np.abs(gpu - ref)
    share = float(np.mean(err > ATOL + RTOL * np.abs(ref)))
    msg = "%s: GPU vs fp64 oracle mean %.4g max %.4g share %.4g; fp32 oracle vs fp64 mean %.4g max %.4g share %.4g" % (
        what, err.mean(), err.max(), share, floor["mean"], floor["max"], floor["share"])
    assert err.mean() <= FLOOR_FACTOR * floor["mean"], msg
    assert err.max() <= FLOOR_FACTOR * floor["max"], msg
    assert share <= FLOOR_FACTOR * floor["share"], msg
