"""GPU parity of the verify pass (C ABI through the binding) against the CPU oracle.

Small models whose oracle runs in seconds but whose matrices still span
several 128-row tiles, several 64-wide k-blocks, more than one KV page and
ragged tails (vocab 1000, blocks of 1..16 tokens, contexts off page
boundaries)."""
import os

import numpy as np
import pytest

import oracle
import synth
from conftest import small_gqa_cfg, small_moe_cfg
from gpu_common import ATOL, RTOL, argmax_mismatches, assert_logits_close, make_model, torch_cuda

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def torch():
    return torch_cuda()


@pytest.fixture(scope="module")
def tiny_model(torch, tiny_cfg, tiny_weights):
    return make_model(tiny_cfg, tiny_weights, draft_plan=oracle.layer_skip_plan(tiny_cfg.n_layers, 0.5))


def reset(m):
    import speculative_decoding_verify_pass_gb300 as sv
    m.kv_set_len(sv.SPEC_CACHE_TARGET, 0)
    if m.draft_plan:
        m.kv_set_len(sv.SPEC_CACHE_DRAFT, 0)


def test_library_exports_and_launches(torch, tiny_model):
    import speculative_decoding_verify_pass_gb300 as sv
    lib = sv.library()
    for name in sv.EXPORTED:
        assert hasattr(lib, name)
    reset(tiny_model)
    tiny_model.prefill(np.arange(20, dtype=np.int32))
    assert tiny_model.launches() > 0


def test_tiny_prefill_verify_logits_match_oracle(torch, tiny_cfg, tiny_oracle, tiny_model, tiny_prompt):
    m, orc = tiny_model, tiny_oracle
    reset(m)
    p = tiny_prompt
    nxt = m.prefill(p[:100])
    oc = orc.new_cache()
    ol, _, _ = orc.forward(oc, orc.full_plan, p[:100], 0, logits_from=99)
    argmax_mismatches([int(nxt.item())], ol)
    for n in (1, 2, 5, 8, 9, 16):
        block = torch.tensor(p[100:100 + n], dtype=torch.int32, device="cuda")
        am, acc, lg, _ = m.verify(block, logits=True)
        ref, _, _ = orc.forward(oc, orc.full_plan, p[100:100 + n], 100)
        assert_logits_close(lg.cpu().numpy(), ref, "tiny n=%d" % n)
        argmax_mismatches(am.cpu().numpy(), ref)
        a = [int(np.argmax(r)) for r in ref]
        assert int(acc.item()) == oracle.accept_len(p[100:100 + n], a)
        m.rollback(0, 100)
        oc.truncate(100)


def test_tiny_greedy_matches_golden(torch, tiny_cfg, tiny_model, tiny_prompt):
    reset(tiny_model)
    m = make_model(tiny_cfg, tiny_model_weights(tiny_cfg))
    got = m.greedy(tiny_prompt, 64)
    want = [int(t) for t in open(os.path.join(GOLDEN, "tiny_greedy.txt")).read().split("\n")[-2].split()]
    assert got == want


_W = {}


def tiny_model_weights(cfg):
    if "tiny" not in _W:
        _W["tiny"] = synth.make_weights(cfg)
    return _W["tiny"]


@pytest.mark.parametrize("frac,gamma", [(0.5, 4), (0.25, 1), (0.25, 5), (0.5, 2)])
def test_tiny_selfspec_equals_greedy(torch, tiny_cfg, tiny_prompt, frac, gamma):
    w = tiny_model_weights(tiny_cfg)
    plan = oracle.layer_skip_plan(tiny_cfg.n_layers, frac)
    m = make_model(tiny_cfg, w, draft_plan=plan)
    greedy = m.greedy(tiny_prompt, 64)
    reset(m)
    out, acc = m.selfspec(tiny_prompt, 64, gamma)
    assert out == greedy
    assert all(0 <= k <= gamma for k in acc)


@pytest.mark.parametrize("gamma", [3, 7])
def test_tiny_full_plan_draft_accepts_all(torch, tiny_cfg, tiny_prompt, gamma):
    w = tiny_model_weights(tiny_cfg)
    m = make_model(tiny_cfg, w, draft_plan=list(range(tiny_cfg.n_layers)))
    greedy = m.greedy(tiny_prompt, 40)
    reset(m)
    out, acc = m.selfspec(tiny_prompt, 40, gamma)
    assert out == greedy
    assert all(k == gamma for k in acc)


def test_verify_rows_equal_decode_steps_bitwise(torch, tiny_cfg, tiny_prompt):
    """Batch invariance: row j of a verify pass equals the one-token decode at
    that position, bit for bit (fixed reduction orders; chunked attention on
    absolute positions)."""
    w = tiny_model_weights(tiny_cfg)
    a = make_model(tiny_cfg, w)
    b = make_model(tiny_cfg, w)
    p = tiny_prompt
    a.prefill(p[:70])
    b.prefill(p[:70])
    block = torch.tensor(p[70:86], dtype=torch.int32, device="cuda")
    am, _, lg, _ = a.verify(block, logits=True)
    for j in range(16):
        amj, _, lgj, _ = b.verify(block[j:j + 1].clone(), logits=True)
        assert torch.equal(lg[j], lgj[0]), j
        assert int(am[j]) == int(amj[0])


@pytest.mark.parametrize("shape", ["gqa-small", "qwen3-4b-1layer"])
def test_grouped_rows_equal_decode_steps_bitwise(torch, shape):
    """Batch invariance with grouped heads: a block of 16 tokens (64 query rows
    per kv head, four row groups) and one of 8 (two row groups) against
    one-token decode steps, bit for bit.  The attention unit splits its work
    differently for 1, 2 and 4 row groups; every row must come out the same."""
    if shape == "gqa-small":
        cfg = small_gqa_cfg()
    else:
        cfg = synth.scaled(synth.qwen3_4b(max_ctx=512), n_layers=1)
    w = synth.make_weights(cfg)
    p = synth.prompt(cfg, 200, stream=5)
    for n in (16, 8):
        a = make_model(cfg, w)
        b = make_model(cfg, w)
        a.prefill(p[:130])
        b.prefill(p[:130])
        block = torch.tensor(p[130:130 + n], dtype=torch.int32, device="cuda")
        am, _, lg, _ = a.verify(block, logits=True)
        for j in range(n):
            amj, _, lgj, _ = b.verify(block[j:j + 1].clone(), logits=True)
            assert torch.equal(lg[j], lgj[0]), (shape, n, j)
            assert int(am[j]) == int(amj[0])
        a.close()
        b.close()


def test_launch_trace_records_every_launch(torch, tiny_cfg, tiny_prompt):
    """spec_trace_*: a traced verify records, per launch, its kind and per-CTA
    stamps in order (entry <= inputs ready <= exit)."""
    import speculative_decoding_verify_pass_gb300 as sv
    w = tiny_model_weights(tiny_cfg)
    m = make_model(tiny_cfg, w)
    m.prefill(tiny_prompt[:40])
    sv.spec_trace_enable(m.h, True)
    m.verify(torch.tensor(tiny_prompt[40:44], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    kinds = list(sv.spec_trace_kinds(m.h))
    tr = sv.spec_trace_read(m.h)
    sv.spec_trace_enable(m.h, False)
    per_layer = [sv.EPI_QKV, 16, 17, sv.EPI_RESID, sv.EPI_SWIGLU, sv.EPI_RESID]
    assert kinds == per_layer * tiny_cfg.n_layers + [sv.EPI_LMHEAD]
    assert tr.shape[1] == len(kinds)
    for l in range(len(kinds)):
        s = tr[:, l, :]
        live = s[s[:, 0] > 0]
        assert len(live) > 0, l
        assert np.all(live[:, 3] >= live[:, 0])
        ready = live[live[:, 1] > 0]
        assert np.all(ready[:, 1] >= ready[:, 0]) and np.all(ready[:, 3] >= ready[:, 1])
    m.close()


def test_rollback_equals_recompute_bitwise(torch, tiny_cfg, tiny_prompt):
    w = tiny_model_weights(tiny_cfg)
    a = make_model(tiny_cfg, w)
    b = make_model(tiny_cfg, w)
    p = tiny_prompt
    a.prefill(p[:50])
    a.verify(torch.tensor(p[50:58], dtype=torch.int32, device="cuda"))
    a.rollback(0, 53)
    b.prefill(p[:53])
    blk = torch.tensor([11, 12, 13], dtype=torch.int32, device="cuda")
    _, _, la, _ = a.verify(blk, logits=True)
    _, _, lb, _ = b.verify(blk.clone(), logits=True)
    assert torch.equal(la, lb)
    assert a.kv_len(0) == 56


def test_kv_cache_matches_oracle(torch, tiny_cfg, tiny_oracle, tiny_prompt):
    w = tiny_model_weights(tiny_cfg)
    m = make_model(tiny_cfg, w)
    p = tiny_prompt[:77]
    m.prefill(p)
    oc = tiny_oracle.new_cache()
    tiny_oracle.forward(oc, tiny_oracle.full_plan, p, 0, logits_from=None)
    for layer in (0, tiny_cfg.n_layers - 1):
        k, v = m.kv_export(0, layer, 77)
        kr = oc.read(layer, 0, 77).reshape(77, tiny_cfg.n_kv_heads, tiny_cfg.head_dim)
        vr = oc.read(layer, 1, 77).reshape(77, tiny_cfg.n_kv_heads, tiny_cfg.head_dim)
        kg, vg = synth.bf16_to_f32(k), synth.bf16_to_f32(v)
        assert np.allclose(kg, kr, atol=ATOL, rtol=RTOL)
        assert np.allclose(vg, vr, atol=ATOL, rtol=RTOL)


def test_kv_load_export_roundtrip(torch, tiny_cfg):
    w = tiny_model_weights(tiny_cfg)
    m = make_model(tiny_cfg, w)
    k = synth.synthetic_kv(tiny_cfg, 2, 200, 0)
    v = synth.synthetic_kv(tiny_cfg, 2, 200, 1)
    m.kv_load(0, 2, k, v)
    k2, v2 = m.kv_export(0, 2, 200)
    assert np.array_equal(k, k2) and np.array_equal(v, v2)


@pytest.mark.parametrize("ctx,n", [(0, 7), (63, 2), (64, 16), (130, 5), (255, 16)])
def test_gqa_ragged_vocab_synthetic_context(torch, ctx, n):
    """4 query heads per kv head, tied LM head, vocab 1000 (ragged last tile),
    contexts loaded as synthetic KV that end inside / at page boundaries."""
    cfg = small_gqa_cfg()
    w = synth.make_weights(cfg)
    m = make_model(cfg, w)
    orc = oracle.Oracle(cfg, w)
    oc = orc.new_cache()
    for l in range(cfg.n_layers):
        k = synth.synthetic_kv(cfg, l, max(ctx, 1), 0)[:ctx]
        v = synth.synthetic_kv(cfg, l, max(ctx, 1), 1)[:ctx]
        if ctx:
            m.kv_load(0, l, k, v)
            oc.load(l, k.reshape(ctx, -1), v.reshape(ctx, -1))
    m.kv_set_len(0, ctx)
    oc.set_len(ctx)
    toks = synth.prompt(cfg, n, stream=ctx)
    am, acc, lg, _ = m.verify(torch.tensor(toks, dtype=torch.int32, device="cuda"), logits=True)
    ref, _, _ = orc.forward(oc, orc.full_plan, toks, ctx)
    assert_logits_close(lg.cpu().numpy(), ref, "gqa ctx=%d n=%d" % (ctx, n))
    argmax_mismatches(am.cpu().numpy(), ref)


def many_kv_cfg():
    """32 kv heads of 2 query heads each.  The attention unit makes about
    SMs / kv heads chunk groups per kv head (5 on 152 SMs), so at contexts of
    several hundred positions each group merges several 128-position chunks:
    the running max, running sum and running O of a group are carried across
    chunks, which the smaller models (one chunk per group) never do."""
    return synth.ModelConfig("gqa-many-kv", 2, 256, 64, 32, 64, 512, 1000, rope_theta=5e5,
                             max_ctx=2048, index=7)


def _chunks_per_group(torch, cfg, total):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    groups = min(-(-sms // cfg.n_kv_heads), cfg.max_ctx // 128)
    return -(-(-(-total // 128)) // groups)


def _load_synthetic_context(m, cfg, ctx, oc=None):
    for l in range(cfg.n_layers):
        k = synth.synthetic_kv(cfg, l, ctx, 0)
        v = synth.synthetic_kv(cfg, l, ctx, 1)
        m.kv_load(0, l, k, v)
        if oc is not None:
            oc.load(l, k.reshape(ctx, -1), v.reshape(ctx, -1))
    m.kv_set_len(0, ctx)
    if oc is not None:
        oc.set_len(ctx)


@pytest.mark.parametrize("ctx,n", [(700, 3), (1000, 16), (1900, 8)])
def test_multichunk_groups_match_oracle(torch, ctx, n):
    """Chunk groups of two and three chunks (running max, sum and O carried
    across chunks, both parities of the per-row state) against the oracle at
    the stated tolerance."""
    cfg = many_kv_cfg()
    assert _chunks_per_group(torch, cfg, ctx + n) >= 2
    w = synth.make_weights(cfg)
    m = make_model(cfg, w)
    orc = oracle.Oracle(cfg, w)
    oc = orc.new_cache()
    _load_synthetic_context(m, cfg, ctx, oc)
    toks = synth.prompt(cfg, n, stream=ctx)
    am, _, lg, _ = m.verify(torch.tensor(toks, dtype=torch.int32, device="cuda"), logits=True)
    ref, _, _ = orc.forward(oc, orc.full_plan, toks, ctx)
    assert_logits_close(lg.cpu().numpy(), ref, "many-kv ctx=%d n=%d" % (ctx, n))
    argmax_mismatches(am.cpu().numpy(), ref)
    m.close()


def test_multichunk_groups_rows_equal_decode_steps_bitwise(torch):
    """Batch invariance where every chunk group merges two chunks: a block of
    16 against one-token decode steps, bit for bit."""
    cfg = many_kv_cfg()
    ctx = 1100
    assert _chunks_per_group(torch, cfg, ctx + 16) >= 2
    w = synth.make_weights(cfg)
    a = make_model(cfg, w)
    b = make_model(cfg, w)
    _load_synthetic_context(a, cfg, ctx)
    _load_synthetic_context(b, cfg, ctx)
    block = torch.tensor(synth.prompt(cfg, 16, stream=3), dtype=torch.int32, device="cuda")
    am, _, lg, _ = a.verify(block, logits=True)
    for j in range(16):
        amj, _, lgj, _ = b.verify(block[j:j + 1].clone(), logits=True)
        assert torch.equal(lg[j], lgj[0]), j
        assert int(am[j]) == int(amj[0])
    a.close()
    b.close()


@pytest.mark.parametrize("hd,kv,ctx,n", [(64, 2, 3000, 5), (64, 2, 4000, 16), (128, 4, 3600, 8)])
def test_merge_of_more_groups_than_its_first_sweep(torch, hd, kv, ctx, n):
    """Few kv heads and a long context: a row has more chunk groups (24, 32,
    29) than the merge kernel loads in its first sweep (20), so the later
    groups go through its batches of eight (one, two and two batches, the
    last one partial), for head dims 64 and 128."""
    cfg = synth.ModelConfig("gqa-long-%d" % hd, 2, 256, 4 * kv, kv, hd, 512, 1000, rope_theta=5e5,
                            max_ctx=4224, index=8)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    groups = min(-(-sms // kv), -(-cfg.max_ctx // 128))
    assert min(groups, -(-(ctx + n) // 128)) > 20
    w = synth.make_weights(cfg)
    m = make_model(cfg, w)
    orc = oracle.Oracle(cfg, w)
    oc = orc.new_cache()
    _load_synthetic_context(m, cfg, ctx, oc)
    toks = synth.prompt(cfg, n, stream=ctx)
    am, _, lg, _ = m.verify(torch.tensor(toks, dtype=torch.int32, device="cuda"), logits=True)
    ref, _, _ = orc.forward(oc, orc.full_plan, toks, ctx)
    assert_logits_close(lg.cpu().numpy(), ref, "long hd=%d ctx=%d n=%d" % (hd, ctx, n))
    argmax_mismatches(am.cpu().numpy(), ref)
    m.close()


def test_moe_small_matches_oracle_and_modes_agree(torch):
    import speculative_decoding_verify_pass_gb300 as sv
    cfg = small_moe_cfg()
    w = synth.make_weights(cfg)
    m = make_model(cfg, w)
    orc = oracle.Oracle(cfg, w)
    p = synth.prompt(cfg, 40)
    m.prefill(p[:30])
    oc = orc.new_cache()
    orc.forward(oc, orc.full_plan, p[:30], 0, logits_from=None)
    results = {}
    for mode in (sv.SPEC_MOE_PER_SLOT, sv.SPEC_MOE_DEDUP):
        m.moe_mode(mode)
        m.kv_set_len(0, 30)
        am, acc, lg, ids = m.verify(torch.tensor(p[30:40], dtype=torch.int32, device="cuda"), logits=True,
                                    expert_ids=True)
        results[mode] = (am.cpu().numpy(), lg.cpu().numpy(), ids.cpu().numpy())
    a, b = results[sv.SPEC_MOE_PER_SLOT], results[sv.SPEC_MOE_DEDUP]
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2])
    gids = a[2]
    ref, rids, _ = orc.forward(oc, orc.full_plan, p[30:40], 30, want_routing=True, forced_ids=np.maximum(gids, 0))
    # the oracle's own (unforced) routing must pick the same experts
    oc2 = orc.new_cache()
    orc.forward(oc2, orc.full_plan, p[:30], 0, logits_from=None)
    _, ids_free, _ = orc.forward(oc2, orc.full_plan, p[30:40], 30, want_routing=True)
    assert np.array_equal(ids_free[1:], gids[1:])
    assert np.all(gids[0] == -1)
    assert_logits_close(a[1], ref, "moe")
    argmax_mismatches(a[0], ref)


def test_argument_errors(torch, tiny_cfg, tiny_model):
    import speculative_decoding_verify_pass_gb300 as sv
    m = tiny_model
    reset(m)
    with pytest.raises(sv.SpecError) as e:
        m.verify(torch.zeros(17, dtype=torch.int32, device="cuda"))
    assert e.value.status == sv.SPEC_ERR_INVALID_ARG
    with pytest.raises(sv.SpecError) as e:
        m.rollback(0, 5)
    assert e.value.status == sv.SPEC_ERR_INVALID_ARG
    with pytest.raises(sv.SpecError):
        m.set_draft_plan([1, 2, 3])        # must keep layer 0
    m.kv_set_len(0, tiny_cfg.max_ctx - 2)
    with pytest.raises(sv.SpecError) as e:
        m.verify(torch.zeros(4, dtype=torch.int32, device="cuda"))
    assert e.value.status == sv.SPEC_ERR_CAPACITY
    reset(m)
    bad = torch.tensor([5, tiny_cfg.vocab + 3], dtype=torch.int32, device="cuda")
    m.verify(bad)
    with pytest.raises(sv.SpecError) as e:
        m.check_error()
    assert e.value.status == sv.SPEC_ERR_INVALID_ARG
    m.check_error()


@pytest.mark.parametrize("graphs", ["1", "0"])
def test_both_launch_paths_match_oracle(torch, tiny_cfg, tiny_oracle, tiny_prompt, monkeypatch, graphs):
    """Passes run either from captured CUDA graphs (default) or as direct
    launches (SPEC_GRAPHS=0); both must match the oracle and the golden greedy."""
    monkeypatch.setenv("SPEC_GRAPHS", graphs)
    w = tiny_model_weights(tiny_cfg)
    m = make_model(tiny_cfg, w, draft_plan=oracle.layer_skip_plan(tiny_cfg.n_layers, 0.5))
    orc = tiny_oracle
    p = tiny_prompt
    m.prefill(p[:90])
    oc = orc.new_cache()
    orc.forward(oc, orc.full_plan, p[:90], 0, logits_from=None)
    for n in (1, 7, 16):
        am, acc, lg, _ = m.verify(torch.tensor(p[90:90 + n], dtype=torch.int32, device="cuda"), logits=True)
        ref, _, _ = orc.forward(oc, orc.full_plan, p[90:90 + n], 90)
        assert_logits_close(lg.cpu().numpy(), ref, "graphs %s n=%d" % (graphs, n))
        argmax_mismatches(am.cpu().numpy(), ref)
        m.rollback(0, 90)
        oc.truncate(90)
    m.check_error()
    want = [int(t) for t in open(os.path.join(GOLDEN, "tiny_greedy.txt")).read().split("\n")[-2].split()]
    m2 = make_model(tiny_cfg, w)
    assert m2.greedy(p, 64) == want
    m2.check_error()
