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
from gpu_common import make_model, torch_cuda

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
