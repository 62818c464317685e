"""The allocation-free accept entry point against the verify pass's own accept.

spec_accept_from_logits_noalloc serves callers that cannot allocate device
memory where they need the accept decision (a process whose pool owns the
device, a serving loop that forbids allocation after warm-up, a thread that
must not stall the device with cudaMalloc).  Its scratch is a fixed array
inside the library.  Here it must reproduce, exactly, the argmax rows and
accept_len that spec_verify_step returned for the same logits, on two calls
in a row (the second reuses the scratch the first left behind).

Self-contained, so it passes alone in a fresh process and after the other
tests; the file name makes pytest collect it last."""
import numpy as np
import pytest

import synth
from conftest import small_gqa_cfg
from gpu_common import make_model, torch_cuda

pytestmark = pytest.mark.gpu


def test_accept_from_logits_noalloc_matches_verify_step():
    torch = torch_cuda()
    import speculative_decoding_verify_pass_gb300 as sv
    cfg = small_gqa_cfg()                       # vocab 1000: a ragged last chunk
    w = synth.make_weights(cfg)
    m = make_model(cfg, w)
    p = synth.prompt(cfg, 48)
    greedy = m.greedy(p[:40], 8)                # the model's own continuation
    # call 1 accepts two drafts then mismatches; call 2 accepts all of them
    blocks = [[greedy[0], greedy[1], greedy[2], (greedy[3] + 1) % cfg.vocab, 5],
              greedy[:7]]
    want_accept = [2, 6]
    for call, blk in enumerate(blocks):
        m.kv_set_len(sv.SPEC_CACHE_TARGET, 40)
        block = torch.tensor(blk, dtype=torch.int32, device="cuda")
        am, acc, lg, _ = m.verify(block, logits=True)
        n = block.numel()
        out_am = torch.full((n,), -7, dtype=torch.int32, device="cuda")
        out_acc = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        sv.spec_accept_from_logits_noalloc(lg, block, out_am, out_acc)
        torch.cuda.synchronize()
        assert torch.equal(out_am, am), (call, out_am.tolist(), am.tolist())
        assert int(out_acc.item()) == int(acc.item()) == want_accept[call]
    m.close()


def test_accept_from_logits_noalloc_matches_host_argmax_at_the_vocab_limit():
    """Logits at the largest vocabulary the fixed scratch holds (2,097,152),
    with planted ties, against numpy's argmax (first maximum): a tie that
    straddles the 2048-entry chunk boundary, one between two chunks far apart,
    one row that is constant, and a maximum in the very last entry.  A second
    call on a small ragged vocabulary follows, reusing the scratch the first
    left behind; neither call allocates through torch's allocator."""
    torch = torch_cuda()
    import speculative_decoding_verify_pass_gb300 as sv
    V = 2097152
    rng = np.random.default_rng(17)
    lg = rng.standard_normal((5, V)).astype(np.float32)
    lg[0, 2047] = lg[0, 2048] = 9.0           # tie across the first chunk boundary -> 2047
    lg[1, 4096] = lg[1, V - 1] = 9.5          # tie between distant chunks -> 4096
    lg[2, :] = 0.25                           # constant row -> 0
    lg[3, V - 1] = 12.0                       # maximum in the last entry
    lg[4, 1_000_003] = 8.0
    want = [int(np.argmax(r)) for r in lg]
    assert want == [2047, 4096, 0, V - 1, 1_000_003]
    cases = [(lg, [7, want[0], want[1], 3, 9]),                 # accepts two drafts
             (rng.standard_normal((3, 1000)).astype(np.float32), None)]
    for call, (logits, blk) in enumerate(cases):
        n = logits.shape[0]
        host_am = [int(np.argmax(r)) for r in logits]
        if blk is None:
            blk = [1] + host_am[:n - 1]                          # accepts every draft
        want_acc = 0
        while want_acc < n - 1 and blk[want_acc + 1] == host_am[want_acc]:
            want_acc += 1
        d_lg = torch.from_numpy(logits).to("cuda")
        d_blk = torch.tensor(blk, dtype=torch.int32, device="cuda")
        out_am = torch.full((n,), -7, dtype=torch.int32, device="cuda")
        out_acc = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated()
        sv.spec_accept_from_logits_noalloc(d_lg, d_blk, out_am, out_acc)
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() == before
        assert out_am.cpu().tolist() == host_am, call
        assert int(out_acc.item()) == want_acc == (2 if call == 0 else n - 1), call


def test_accept_from_logits_noalloc_rejects_sizes_beyond_its_scratch():
    torch = torch_cuda()
    import speculative_decoding_verify_pass_gb300 as sv
    lg = torch.zeros((17, 8), dtype=torch.float32, device="cuda")
    blk = torch.zeros(17, dtype=torch.int32, device="cuda")
    out = torch.zeros(17, dtype=torch.int32, device="cuda")
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        sv.spec_accept_from_logits_noalloc(lg, blk, out, acc)
    assert e.value.status == sv.SPEC_ERR_INVALID_ARG
    big = torch.zeros((1, 2097153), dtype=torch.float32, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        sv.spec_accept_from_logits_noalloc(big, blk[:1], out[:1], acc)
    assert e.value.status == sv.SPEC_ERR_INVALID_ARG
    assert b"2097152" in sv.library().spec_last_error()
    # the binding refuses buffers the kernels would read or write past
    for bad in (lg.to(torch.bfloat16), lg.t(), lg.cpu()):
        with pytest.raises(sv.SpecError) as e:
            sv.spec_accept_from_logits_noalloc(bad, blk, out, acc)
        assert e.value.status == sv.SPEC_ERR_INVALID_ARG
    small = torch.zeros((4, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(sv.SpecError) as e:
        sv.spec_accept_from_logits_noalloc(small, blk[:3], out, acc)
    assert e.value.status == sv.SPEC_ERR_INVALID_ARG
