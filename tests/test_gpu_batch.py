"""Batched sequences: one verify pass over the blocks of several independent
sequences, each with its own cache (LayerSkip summary, "Critical
Assessment": in batched inference one verify pass serves several sequences,
which raises the flops per weight byte read).

Every sequence's rows must equal, bit for bit, a single-sequence verify of
the same block on the same cache (the GEMM columns, attention units and
merges of different sequences never mix), the appended keys/values too, and
each sequence's length must follow the greedy rollback rule.  The logits are
also checked against the oracle per sequence."""
import numpy as np
import pytest

import oracle
import synth
from conftest import small_gqa_cfg, small_moe_cfg
from gpu_common import argmax_mismatches, assert_logits_close, make_model, torch_cuda

pytestmark = pytest.mark.gpu


def _contexts(cfg, lens):
    out = []
    for q, ctx in enumerate(lens):
        kv = []
        for l in range(cfg.n_layers):
            k = synth.synthetic_kv(cfg, l, max(ctx, 1), 2 * q)[:ctx]
            v = synth.synthetic_kv(cfg, l, max(ctx, 1), 2 * q + 1)[:ctx]
            kv.append((k, v))
        out.append(kv)
    return out


def _load_single(m, kv, ctx):
    for l, (k, v) in enumerate(kv):
        if ctx:
            m.kv_load(0, l, k, v)
    m.kv_set_len(0, ctx)


@pytest.mark.parametrize("cfgname,lens,n", [
    ("gqa-small", [0, 63, 130, 255], 4),
    ("gqa-small", [70, 1, 200], 5),
    ("gqa-small", [5] * 16, 1),
    ("gqa-small", [129, 64], 8),
    ("moe-small", [30, 91], 6),
])
def test_batched_rows_equal_single_sequence_verify_bitwise(cfgname, lens, n):
    torch = torch_cuda()
    cfg = small_gqa_cfg() if cfgname == "gqa-small" else small_moe_cfg()
    w = synth.make_weights(cfg)
    nseq = len(lens)
    ctxs = _contexts(cfg, lens)
    blocks = np.stack([synth.prompt(cfg, n, stream=20 + q) for q in range(nseq)]).astype(np.int32)
    single = make_model(cfg, w)
    ref = []
    for q in range(1, nseq, 2):           # odd sequences accept at least their first two drafts
        for j in range(min(2, n - 1)):
            _load_single(single, ctxs[q], lens[q])
            am, _, _, _ = single.verify(torch.tensor(blocks[q], dtype=torch.int32, device="cuda"))
            blocks[q, j + 1] = am.cpu().numpy()[j]
    for q in range(nseq):
        _load_single(single, ctxs[q], lens[q])
        am, acc, lg, _ = single.verify(torch.tensor(blocks[q], dtype=torch.int32, device="cuda"), logits=True)
        kvs = [single.kv_export(0, l, lens[q] + n) for l in range(cfg.n_layers)]
        ref.append((am.cpu().numpy(), int(acc.item()), lg.cpu().numpy(), kvs))
    single.check_error()
    single.close()

    m = make_model(cfg, w)
    m.batch_reserve(nseq)
    for q in range(nseq):
        for l, (k, v) in enumerate(ctxs[q]):
            if lens[q]:
                m.batch_kv_load(q, l, k, v)
        m.batch_set_len(q, lens[q])
    am, acc, lg = m.verify_batch(torch.tensor(blocks, dtype=torch.int32, device="cuda"), logits=True)
    m.check_error()
    am, acc, lg = am.cpu().numpy(), acc.cpu().numpy(), lg.cpu().numpy()
    for q in range(nseq):
        ram, racc, rlg, rkv = ref[q]
        assert np.array_equal(lg[q * n:(q + 1) * n], rlg), "sequence %d logits" % q
        assert np.array_equal(am[q], ram) and acc[q] == racc, q
        if q % 2 == 1:
            assert acc[q] >= min(2, n - 1)
        assert m.batch_len(q) == lens[q] + racc + 1
        for l in range(cfg.n_layers):
            k, v = m.batch_kv_export(q, l, lens[q] + n)
            assert np.array_equal(k, rkv[l][0]) and np.array_equal(v, rkv[l][1]), (q, l)
    m.close()


def test_batched_logits_match_oracle_per_sequence():
    torch = torch_cuda()
    cfg = small_gqa_cfg()
    w = synth.make_weights(cfg)
    lens, n = [33, 140, 0], 5
    ctxs = _contexts(cfg, lens)
    blocks = np.stack([synth.prompt(cfg, n, stream=40 + q) for q in range(3)]).astype(np.int32)
    m = make_model(cfg, w)
    m.batch_reserve(4)
    for q in range(3):
        for l, (k, v) in enumerate(ctxs[q]):
            if lens[q]:
                m.batch_kv_load(q, l, k, v)
        m.batch_set_len(q, lens[q])
    am, acc, lg = m.verify_batch(torch.tensor(blocks, dtype=torch.int32, device="cuda"), logits=True)
    m.check_error()
    orc = oracle.Oracle(cfg, w)
    for q in range(3):
        oc = orc.new_cache()
        for l, (k, v) in enumerate(ctxs[q]):
            if lens[q]:
                oc.load(l, k.reshape(lens[q], -1), v.reshape(lens[q], -1))
        oc.set_len(lens[q])
        ref, _, _ = orc.forward(oc, orc.full_plan, blocks[q].tolist(), lens[q])
        assert_logits_close(lg[q * n:(q + 1) * n].cpu().numpy(), ref, "batched sequence %d" % q)
        flagged = argmax_mismatches(am[q].cpu().numpy(), ref)
        if not flagged:
            assert int(acc[q]) == oracle.accept_len(blocks[q].tolist(), [int(np.argmax(r)) for r in ref])
    m.close()


def test_batch_errors_and_repeated_passes():
    torch = torch_cuda()
    import speculative_decoding_verify_pass_gb300 as sv
    cfg = small_gqa_cfg()
    w = synth.make_weights(cfg)
    m = make_model(cfg, w)
    blk = torch.zeros((2, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        m.verify_batch(blk)                           # nothing reserved
    assert e.value.status == sv.SPEC_ERR_INVALID_ARG
    m.batch_reserve(2)
    with pytest.raises(sv.SpecError) as e:
        m.batch_reserve(2)
    assert e.value.status == sv.SPEC_ERR_STATE
    with pytest.raises(sv.SpecError) as e:
        m.verify_batch(torch.zeros((3, 4), dtype=torch.int32, device="cuda"))
    assert e.value.status == sv.SPEC_ERR_INVALID_ARG
    with pytest.raises(sv.SpecError) as e:
        m.verify_batch(torch.zeros((2, 9), dtype=torch.int32, device="cuda"))   # 18 rows
    assert e.value.status == sv.SPEC_ERR_INVALID_ARG
    m.batch_set_len(0, 0)
    m.batch_set_len(1, cfg.max_ctx - 3)
    with pytest.raises(sv.SpecError) as e:
        m.verify_batch(blk)
    assert e.value.status == sv.SPEC_ERR_CAPACITY
    # repeated passes advance each sequence by its own accept + 1
    m.batch_set_len(1, 10)
    toks = torch.tensor(np.stack([synth.prompt(cfg, 4, stream=q) for q in range(2)]), dtype=torch.int32, device="cuda")
    total = [0, 10]
    for _ in range(3):
        _, acc, _ = m.verify_batch(toks)
        a = acc.cpu().numpy()
        total = [total[q] + int(a[q]) + 1 for q in range(2)]
    m.check_error()
    assert [m.batch_len(q) for q in range(2)] == total
    # the single-sequence cache is untouched by batched passes
    assert m.kv_len(0) == 0
    m.close()
