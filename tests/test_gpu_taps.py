"""Hidden-state taps of the verify pass (the target hidden states from which
the mlx-dflash README, "Architecture", builds the draft's context features)
against the oracle's residual stream after the same layers.

The tap is the fp32 residual the next layer's norm reads; the oracle keeps
it in fp32 too, so the comparison is the same one as the oracle's own pin
against the float64 library path: largest error within 2e-2 and mean error
within 2e-3 of the largest magnitude.  Taps must not perturb the pass (logits
bitwise equal with and without them), must leave rows >= n untouched, and
must agree between the captured-graph and direct-launch paths."""
import numpy as np
import pytest

import oracle
import synth
from conftest import small_gqa_cfg, small_moe_cfg
from gpu_common import ATOL, RTOL, TIE_GAP, make_model, torch_cuda

pytestmark = pytest.mark.gpu


def _assert_hidden_close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    scale = float(np.max(np.abs(ref)))
    assert np.max(err) <= 2e-2 * scale and np.mean(err) <= 2e-3 * scale, (
        "%s: max err %.3g mean err %.3g scale %.3g" % (what, np.max(err), np.mean(err), scale))


def _load_context(m, orc, oc, cfg, ctx):
    for l in range(cfg.n_layers):
        k = synth.synthetic_kv(cfg, l, max(ctx, 1), 0)[:ctx]
        v = synth.synthetic_kv(cfg, l, max(ctx, 1), 1)[:ctx]
        if ctx:
            m.kv_load(0, l, k, v)
            oc.load(l, k.reshape(ctx, -1), v.reshape(ctx, -1))
    m.kv_set_len(0, ctx)
    oc.set_len(ctx)


@pytest.mark.parametrize("shape,ctx,n", [("gqa-small", 130, 16), ("gqa-small", 63, 3), ("tiny", 70, 5)])
def test_dense_taps_match_oracle_hidden_states(shape, ctx, n):
    torch = torch_cuda()
    cfg = small_gqa_cfg() if shape == "gqa-small" else synth.tiny()
    w = synth.make_weights(cfg)
    m = make_model(cfg, w)
    orc = oracle.Oracle(cfg, w)
    oc = orc.new_cache()
    _load_context(m, orc, oc, cfg, ctx)
    toks = synth.prompt(cfg, n, stream=ctx + 1)
    blk = torch.tensor(toks, dtype=torch.int32, device="cuda")
    _, _, lg_off, _ = m.verify(blk, logits=True)
    layers = list(range(cfg.n_layers))[::-1]          # any order: slot t holds layers[t]
    taps = m.set_taps(layers)
    m.kv_set_len(0, ctx)
    _, _, lg_on, _ = m.verify(blk, logits=True)
    m.check_error()
    assert torch.equal(lg_on, lg_off)
    got = taps.cpu().numpy()
    assert not np.any(got[:, n:, :]), "rows beyond the block were written"
    hid = np.zeros((cfg.n_layers, n, cfg.d_model), np.float32)
    orc.forward(oc, orc.full_plan, toks, ctx, logits_from=None, hidden=hid)
    for t, l in enumerate(layers):
        _assert_hidden_close(got[t, :n], hid[l], "%s layer %d" % (shape, l))
    m.set_taps([])
    m.close()


def test_moe_taps_match_oracle_under_the_gpu_routing():
    torch = torch_cuda()
    cfg = small_moe_cfg()
    w = synth.make_weights(cfg)
    m = make_model(cfg, w)
    orc = oracle.Oracle(cfg, w)
    p = synth.prompt(cfg, 40)
    m.prefill(p[:30])
    oc = orc.new_cache()
    orc.forward(oc, orc.full_plan, p[:30], 0, logits_from=None)
    layers = [0, cfg.n_layers - 1]                    # a dense layer and a MoE layer
    taps = m.set_taps(layers)
    m.kv_set_len(0, 30)
    _, _, _, ids = m.verify(torch.tensor(p[30:40], dtype=torch.int32, device="cuda"), expert_ids=True)
    m.check_error()
    got = taps.cpu().numpy()
    hid = np.zeros((cfg.n_layers, 10, cfg.d_model), np.float32)
    orc.forward(oc, orc.full_plan, p[30:40], 30, logits_from=None, want_routing=True,
                forced_ids=np.maximum(ids.cpu().numpy(), 0), hidden=hid)
    for t, l in enumerate(layers):
        _assert_hidden_close(got[t, :10], hid[l], "moe layer %d" % l)
    m.close()


def test_full_width_tap_matches_oracle():
    """Llama-3.1-8B width (d 4096, 32/8 heads, F 14336), one layer, synthetic
    context of 128 positions, a block of 16."""
    torch = torch_cuda()
    ctx, n = 128, 16
    cfg = synth.scaled(synth.PRESETS["llama-3.1-8b"](max_ctx=ctx + 64), n_layers=1)
    w = synth.make_weights(cfg)
    m = make_model(cfg, w)
    orc = oracle.Oracle(cfg, w)
    oc = orc.new_cache()
    _load_context(m, orc, oc, cfg, ctx)
    taps = m.set_taps([0])
    toks = synth.prompt(cfg, n, stream=3)
    m.verify(torch.tensor(toks, dtype=torch.int32, device="cuda"))
    m.check_error()
    hid = np.zeros((1, n, cfg.d_model), np.float32)
    orc.forward(oc, orc.full_plan, toks, ctx, logits_from=None, hidden=hid)
    _assert_hidden_close(taps.cpu().numpy()[0, :n], hid[0], "llama width layer 0")
    m.close()


def test_taps_graph_and_direct_paths_agree_and_errors(monkeypatch):
    torch = torch_cuda()
    import speculative_decoding_verify_pass_gb300 as sv
    cfg = small_gqa_cfg()
    w = synth.make_weights(cfg)
    toks = torch.tensor(synth.prompt(cfg, 9, stream=5), dtype=torch.int32, device="cuda")
    out = {}
    for graphs in ("1", "0"):
        monkeypatch.setenv("SPEC_GRAPHS", graphs)
        m = make_model(cfg, w)
        taps = m.set_taps([1, 2])
        for _ in range(3):                       # replayed sequences write the taps every time
            taps.zero_()
            m.kv_set_len(0, 0)
            m.verify(toks)
        m.check_error()
        out[graphs] = taps.clone()
        with pytest.raises(sv.SpecError) as e:
            sv.spec_set_taps(m.h, [1, 1], taps)
        assert e.value.status == sv.SPEC_ERR_INVALID_ARG
        with pytest.raises(sv.SpecError) as e:
            sv.spec_set_taps(m.h, [cfg.n_layers], taps)
        assert e.value.status == sv.SPEC_ERR_INVALID_ARG
        # a rejected call leaves the previous taps in place
        taps.zero_()
        m.kv_set_len(0, 0)
        m.verify(toks)
        m.check_error()
        assert torch.equal(taps, out[graphs])
        # switched off: nothing is written
        m.set_taps([])
        taps.zero_()
        m.kv_set_len(0, 0)
        m.verify(toks)
        m.check_error()
        assert not torch.any(taps)
        m.close()
    assert torch.any(out["1"]) and torch.equal(out["1"], out["0"])


# ----------------------------------------------------------------------------
# Block-draft conditioning (context append) and the block pass over it
# ----------------------------------------------------------------------------
def _identity_bits(d):
    eye = np.zeros((d, d), np.uint16)
    eye[np.arange(d), np.arange(d)] = 0x3F80          # bf16 1.0
    return eye


def test_context_append_of_embeddings_equals_prefill_layer0_bitwise():
    """fc the identity and taps holding token embeddings: the appended layer-0
    keys and values are bitwise those the prefill of the same tokens writes
    (same operand writer, same QKV GEMM)."""
    torch = torch_cuda()
    cfg = small_gqa_cfg()
    w = synth.make_weights(cfg)
    toks = synth.prompt(cfg, 11, stream=4)
    a = make_model(cfg, w)
    a.set_context_fc(_identity_bits(cfg.d_model))
    taps = torch.zeros((1, 16, cfg.d_model), dtype=torch.float32, device="cuda")
    taps[0, :11] = torch.from_numpy(synth.bf16_to_f32(w.embed[toks])).to("cuda")
    a.context_append(taps, 11)
    a.check_error()
    assert a.kv_len(0) == 11
    b = make_model(cfg, w)
    b.prefill(toks)
    ka, va = a.kv_export(0, 0, 11)
    kb, vb = b.kv_export(0, 0, 11)
    assert np.array_equal(ka, kb) and np.array_equal(va, vb)
    a.close()
    b.close()


@pytest.mark.parametrize("shape", ["gqa-small", "qwen3-8b-2layer"])
def test_context_append_and_block_pass_match_oracle(shape):
    """Random fc over three taps; two appends (7 then 9 positions) on top of a
    synthetic context; every layer's appended keys/values against the oracle's
    context append, then a block of 16 ([last, mask x 15]) over that cache:
    logits against the oracle forward on the oracle's cache.  At Qwen3-8B
    width the reference is the fp64-accumulating oracle and the bound the
    fp32 oracle's own deviation from it on the same inputs (the floor rule of
    the full-size tests, computed here rather than stored)."""
    torch = torch_cuda()
    from gpu_common import argmax_mismatches, assert_logits_close, assert_within_floor
    if shape == "gqa-small":
        cfg = small_gqa_cfg()
    else:
        cfg = synth.scaled(synth.PRESETS["qwen3-8b"](max_ctx=256), n_layers=2)
    w = synth.make_weights(cfg)
    d, n_in, ctx = cfg.d_model, 3, 70
    fc = synth.normal_bf16((d, n_in * d), 31, 2)
    rng = np.random.default_rng(5)
    m = make_model(cfg, w)
    m.set_context_fc(fc)
    orc = oracle.Oracle(cfg, w)
    oc = orc.new_cache()
    _load_context(m, orc, oc, cfg, ctx)
    wide = shape != "gqa-small"
    if wide:
        o64 = oracle.Oracle(cfg, w, acc64=True)
        oc64 = o64.new_cache()
        for l in range(cfg.n_layers):
            oc64.load(l, synth.synthetic_kv(cfg, l, ctx, 0).reshape(ctx, -1),
                      synth.synthetic_kv(cfg, l, ctx, 1).reshape(ctx, -1))
        oc64.set_len(ctx)
    for rows in (7, 9):
        taps = rng.standard_normal((n_in, 16, d)).astype(np.float32)
        m.context_append(torch.from_numpy(taps).to("cuda"), rows)
        orc.context_append(oc, fc, taps, rows)
        if wide:
            o64.context_append(oc64, fc, taps, rows)
    m.check_error()
    total = ctx + 16
    assert m.kv_len(0) == total and oc.len == total
    for l in range(cfg.n_layers):
        kg, vg = m.kv_export(0, l, total)
        for which, g in ((0, kg), (1, vg)):
            got = synth.bf16_to_f32(g.reshape(total, -1)[ctx:]).astype(np.float64)
            ref = oc.read(l, which, total)[ctx:].astype(np.float64)
            err = np.abs(got - ref)
            scale = float(np.max(np.abs(ref)))
            assert np.max(err) <= 2e-2 * scale and np.mean(err) <= 2e-3 * scale, (shape, l, which)
    mask = cfg.vocab - 1
    block = [int(synth.prompt(cfg, 1, stream=9)[0])] + [mask] * 15
    am, _, lg, _ = m.verify(torch.tensor(block, dtype=torch.int32, device="cuda"), logits=True)
    m.check_error()
    ref, _, _ = orc.forward(oc, orc.full_plan, block, total)
    if wide:
        ref64, _, _ = o64.forward(oc64, o64.full_plan, block, total)
        e = np.abs(ref.astype(np.float64) - ref64)
        floor = dict(mean=float(e.mean()), max=float(e.max()),
                     share=float(np.mean(e > ATOL + RTOL * np.abs(ref64))))
        assert_within_floor(lg.cpu().numpy(), ref64, floor, "block pass %s" % shape)
        # a near tie is a top-two margin the fp32 arithmetic itself may reorder
        argmax_mismatches(am.cpu().numpy(), ref64, tie_gap=max(TIE_GAP, 2.0 * floor["max"]))
    else:
        assert_logits_close(lg.cpu().numpy(), ref, "block pass %s" % shape)
        argmax_mismatches(am.cpu().numpy(), ref)
    m.rollback(0, total)                   # the block's own keys/values are dropped
    assert m.kv_len(0) == total
    m.close()


def test_context_append_errors():
    torch = torch_cuda()
    import speculative_decoding_verify_pass_gb300 as sv
    cfg = small_gqa_cfg()
    w = synth.make_weights(cfg)
    m = make_model(cfg, w)
    taps = torch.zeros((2, 16, cfg.d_model), dtype=torch.float32, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        m.context_append(taps, 4)                      # no fc yet
    assert e.value.status == sv.SPEC_ERR_STATE
    m.set_context_fc(synth.normal_bf16((cfg.d_model, 2 * cfg.d_model), 3, 1))
    with pytest.raises(sv.SpecError) as e:
        m.set_context_fc(synth.normal_bf16((cfg.d_model, 2 * cfg.d_model), 3, 1))
    assert e.value.status == sv.SPEC_ERR_STATE
    for bad in (0, 17):
        with pytest.raises(sv.SpecError) as e:
            m.context_append(taps, bad)
        assert e.value.status == sv.SPEC_ERR_INVALID_ARG
    m.kv_set_len(0, cfg.max_ctx - 3)
    with pytest.raises(sv.SpecError) as e:
        m.context_append(taps, 4)
    assert e.value.status == sv.SPEC_ERR_CAPACITY
    m.context_append(taps, 3)
    m.check_error()
    assert m.kv_len(0) == cfg.max_ctx
    m.close()
