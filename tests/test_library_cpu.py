"""CPU checks of the C ABI library and the host-side logic (no GPU needed).

The library cross-compiles for sm_103a here and loads without a device;
every symbol declared in include/spec.h must be exported.  No compute call is
made."""
import ctypes
import os
import re

import pytest

import synth
from oracle import closed_forms as cf

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "spec.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verify_pass_gb300 import _build
    path = _build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary_calls():
    names = declared_symbols()
    for required in ("spec_model_create", "spec_prefill", "spec_draft_step", "spec_verify_step", "spec_kv_rollback",
                     "spec_moe_mode", "spec_model_destroy", "spec_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_lists_every_declared_symbol():
    import speculative_decoding_verify_pass_gb300 as sv
    assert sorted(sv.EXPORTED) == declared_symbols()


def test_argument_errors_need_no_device(lib):
    """Host-side validation answers before any CUDA call."""
    import speculative_decoding_verify_pass_gb300 as sv
    L = sv.library()
    assert L.spec_verify_step(None, None, 4, None, None, None, None, None) == sv.SPEC_ERR_INVALID_ARG
    assert L.spec_kv_rollback(None, 0, 3) == sv.SPEC_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert L.spec_model_create(None, None, None, 0, None, ctypes.byref(h)) == sv.SPEC_ERR_INVALID_ARG
    assert b"null config" in L.spec_last_error()
    bad = sv._config_c(synth.scaled(synth.tiny(), d_model=200))
    assert L.spec_model_create(ctypes.byref(bad), None, None, 0, None, ctypes.byref(h)) == sv.SPEC_ERR_INVALID_ARG
    assert b"multiple of 128" in L.spec_last_error()
    bad = sv._config_c(synth.scaled(synth.tiny(), head_dim=96))
    assert L.spec_model_create(ctypes.byref(bad), None, None, 0, None, ctypes.byref(h)) == sv.SPEC_ERR_INVALID_ARG
    # the expert kernels hold at most two shared experts per MoE layer as work items
    bad = sv._config_c(synth.scaled(synth.moe_v2lite(), n_shared_experts=3))
    assert L.spec_model_create(ctypes.byref(bad), None, None, 0, None, ctypes.byref(h)) == sv.SPEC_ERR_INVALID_ARG
    assert b"n_shared_experts must be 0..2" in L.spec_last_error()


def test_layer_skip_plan_matches_hand_worked_table():
    import speculative_decoding_verify_pass_gb300 as sv
    rows = [l.split() for l in open(os.path.join(ROOT, "tests", "golden", "skip_sets.txt"))
            if l.strip() and l[0] != "#"]
    for L, f, a, b in rows:
        keep = sv.layer_skip_plan(int(L), float(f))
        assert [i for i in range(int(L)) if i not in keep] == list(range(int(a), int(b) + 1))


def test_bench_byte_model_matches_closed_form():
    import bench
    for c in (synth.qwen3_4b(), synth.llama31_8b(), synth.qwen3_8b(), synth.tiny()):
        for n, ctx in ((1, 0), (4, 2048), (16, 4096)):
            assert bench.pass_bytes(c, n, ctx) == cf.pass_bytes(c, n, ctx).total


def test_product_path_does_not_import_the_oracle():
    """The CUDA path and the binding must never reach the oracle."""
    pkg = os.path.join(ROOT, "speculative_decoding_verify_pass_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower().replace("oracles", ""), f


def test_step_model_matches_oracle_closed_forms():
    """The benchmark's product-side step model against the oracle's closed forms."""
    import numpy as np
    from speculative_decoding_verify_pass_gb300 import stepmodel as sm
    for c in (synth.qwen3_4b(), synth.llama31_8b(), synth.qwen3_8b(), synth.tiny()):
        for n, ctx in ((1, 0), (4, 2048), (16, 4096)):
            assert sm.pass_bytes(c, n, ctx) == cf.pass_bytes(c, n, ctx).total
    for a in np.linspace(0, 1, 22):
        for g in range(0, 16):
            assert abs(sm.tokens_per_verify(a, g) - cf.expected_tokens(a, g)) < 1e-12
    for n in range(1, 17):
        assert abs(sm.union_size_expected(n, 64, 6) - cf.expected_union(n, 64, 6)) < 1e-9
    tv = lambda n: 1.0 + 0.05 * (n - 1)
    for a in np.linspace(0, 1, 22):
        assert sm.best_gamma(a, tv, 0.1, range(16)) == cf.best_draft_length(a, tv, 0.1, range(16))
    assert abs(sm.mean_accept_truncated(sm.alpha_for_mean_accept(6.0, 15), 15) - 6.0) < 1e-9
    assert abs(sm.alpha_for_mean_accept(6.0, 15) - 0.87358) < 1e-4
    assert abs(sm.alpha_for_mean_accept(9.0, 15) - 0.93293) < 1e-4
    moe = synth.moe_v2lite()
    assert sm.expert_bytes(moe) == 3 * 1408 * 2048 * 2


def test_step_model_predictions_from_fitted_bandwidths():
    """The MoE suite's prediction helpers: the saving and its bound, the
    crossover they imply, and a monotone best-draft-length staircase from
    predicted verify times."""
    import numpy as np
    from speculative_decoding_verify_pass_gb300 import stepmodel as sm
    bw, err = sm.fit_bandwidth([10.0, 10.0, 10.0], [1.0, 1.25, 0.8])
    assert abs(bw - (10.0 + 8.0 + 12.5) / 3) < 1e-12 and abs(err - 2.25 / bw) < 1e-12
    # the saving equals the time identity, and the bound covers the saving
    # under any bandwidths within the stated errors
    bps, bdd = [3.0, 5.0], [2.0, 3.0]
    s, bound = sm.dedup_saving(bps, bdd, 2.0, 1.5, 0.1, 0.05)
    assert abs(s - (8.0 / 2.0 - 5.0 / 1.5)) < 1e-12
    for f_ps in (0.9, 1.0, 1.1):
        for f_dd in (0.95, 1.0, 1.05):
            s2 = 8.0 / (2.0 * f_ps) - 5.0 / (1.5 * f_dd)
            assert abs(s2 - s) <= bound + 1e-12
    # crossover: the first pass size whose saving is positive is the first
    # whose byte share is below the bandwidth ratio
    ns = range(1, 9)
    bw_ps, bw_dd = 1.0, 0.6
    u = [1.0, 0.8, 0.7, 0.62, 0.55, 0.5, 0.47, 0.45]
    sav = [sm.dedup_saving([1.0], [ui], bw_ps, bw_dd, 0.0, 0.0)[0] for ui in u]
    assert sm.first_win(ns, u, [bw_dd / bw_ps] * 8) == next(n for n, v in zip(ns, sav) if v > 0) == 5
    # predicted verify times: the plain step is reproduced; the staircase is monotone
    tv = sm.predicted_verify_times(1000.0, lambda n: 200.0 + 40.0 * (n - 1), ns)
    assert tv[1] == 1000.0 and tv[8] == 1000.0 + 280.0
    st = sm.gamma_staircase(np.linspace(0.0, 1.0, 22), lambda n: tv[n], 300.0, range(0, 8))
    assert st[0] == 0 and all(b >= a for a, b in zip(st, st[1:]))


def test_step_model_affine_fit():
    """t = t0 + bytes / B recovered from exact points; the relative error is
    the largest residual; the summed model time of several operations."""
    from speculative_decoding_verify_pass_gb300 import stepmodel as sm
    b = [1e9, 2e9, 3e9, 4e9]
    t0, bw, err = sm.fit_time_model(b, [6e-4 + x / 2e12 for x in b])
    assert abs(t0 - 6e-4) < 1e-12 and abs(bw - 2e12) / 2e12 < 1e-9 and err < 1e-9
    t0, bw, err = sm.fit_time_model(b, [1.0e-3, 1.7e-3, 2.0e-3, 2.6e-3])
    resid = [abs(t - t0 - x / bw) / t for x, t in zip(b, [1.0e-3, 1.7e-3, 2.0e-3, 2.6e-3])]
    assert abs(err - max(resid)) < 1e-12 and err > 0.01
    assert abs(sm.model_time(1e-4, 1e12, [1e9, 3e9]) - (2e-4 + 4e-3)) < 1e-15
