"""Benchmark of the speculative-decoding verify pass on one GB300 (or N replicas).

Default step (--workload geometric): one verify cycle of the Llama-3.1-8B-
shaped target (random-init bf16 weights) at KV context 4096 (seeded
synthetic keys and values): a block of n tokens (default 8: the last accepted
token and 7 drafts) through all 32 layers with argmax and the cumulative-
product accept, then the device-side rollback.  The drafts are seeded
corruptions of the target's own greedy continuation, each draft clean with
probability alpha (default 0.7), so acceptance is geometric:
P(accept_len >= j) = alpha^j.  Which drafts are clean depends only on the
seeded stream, so the cycle schedule (block start, accept length) is fixed
before the run and the device's accept lengths are checked against it.  The
loop stays on the device; each block is copied into the verify's input
buffer on the device.

--workload selfspec keeps the earlier step: one greedy self-speculative cycle
of the Qwen3-4B-shaped target at context 2048 (gamma draft steps over the
middle-skip plan, verify n = gamma+1, accept, rollback of both caches).

Printed JSON line: accepted tokens/s (the MLX post's and the DFlash README's
throughput metric), the verify pass's time and HBM bandwidth against 8 TB/s
for every block size up to the headline one, a roofline entry for the
streaming GEMM (the dominant kernel) from an in-pipeline launch trace, an
end-to-end figure through the host-driven API with pinned host copies, the
oracle's rate on the host cores, and the SM clocks seen during the timed
region.

    python bench.py [--steps K] [--warmup W] [--n 8] [--alpha 0.7]
    python bench.py --workload selfspec [--gamma 3] [--skip 0.5]
    python bench.py --impl reference     # the CPU oracle on the same workload
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verify-pass time & HBM GB/s (% of 8 TB/s) vs draft length; accepted tok/s"
NOMINAL_HBM = 8000.0  # GB/s


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


GEMM_SOURCES = ("common.cuh", "internal.h", "gemm_core.cuh", "gemm.cu")


def traffic_profile(model):
    """The committed ncu capture of the streaming GEMM's DRAM bytes for a model shape."""
    return os.path.join(ROOT, "profiles", "gemm_kernel_dram_%s.txt" % model)


def gemm_source_sha256():
    """Digest of the sources the streaming GEMM is compiled from."""
    import hashlib
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "speculative_decoding_verify_pass_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def ncu_traffic(launches_by_kind, cfg, args):
    """DRAM bytes (read + write) per GEMM launch from the committed ncu
    capture, averaged over this run's launch mix by epilogue kind; None when
    the capture is of another workload or of other GEMM sources.  The capture
    may be of the model truncated to its first layers: the launches have the
    same matrix shapes, so the same bytes per launch of each kind."""
    path = traffic_profile(cfg.name)
    if not os.path.exists(path):
        return None, "no ncu capture committed for this model"
    per_kind, digest, model = {}, None, None
    for line in open(path):
        f = line.split()
        if len(f) >= 2 and f[0] == "source_sha256":
            digest = f[1]
        elif len(f) >= 2 and f[0] == "model":
            model = f[1]
        elif len(f) == 6 and f[0] == "kind":
            per_kind[int(f[1])] = float(f[3]) + float(f[5])
    if model != cfg.name:
        return None, "ncu capture is of another model"
    if digest != gemm_source_sha256():
        return None, "GEMM sources changed since the ncu capture"
    n = sum(launches_by_kind.values())
    if n == 0 or any(k not in per_kind for k, c in launches_by_kind.items() if c):
        return None, "ncu capture lacks a launch kind of this run"
    tot = sum(per_kind[k] * c for k, c in launches_by_kind.items() if c)
    return round(tot / n), os.path.relpath(path, ROOT)


def pass_bytes(cfg, n, ctx, plan=None):
    from speculative_decoding_verify_pass_gb300 import stepmodel
    return stepmodel.pass_bytes(cfg, n, ctx, plan)


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 100

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        """Start sampling; returns once the first sample has arrived (or after
        two seconds), so that the timed region that follows is covered."""
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms",
               str(self.PERIOD_MS)]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 2.0:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t_begin=None, t_end=None):
        """Stop sampling and summarise the samples that arrived between
        t_begin and t_end (host seconds; one period of slack after t_end).
        With no sample in that window every sample is used, and the line says
        so."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(2 * self.PERIOD_MS / 1e3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return summarize_clock_lines(self.lines, t_begin, t_end, self.PERIOD_MS / 1e3)


def _sample_time(stamp, arrival):
    """A sample's own time (nvidia-smi's local-time stamp) as host seconds,
    else the time its line was read (the pipe may deliver lines late)."""
    import datetime
    try:
        return datetime.datetime.strptime(stamp, "%Y/%m/%d %H:%M:%S.%f").timestamp()
    except ValueError:
        return arrival


def summarize_clock_lines(lines, t_begin=None, t_end=None, slack=0.05):
    """Median SM clock, maximum SM clock and the throttle reasons seen, from
    (arrival time, nvidia-smi csv line) pairs of the fields in
    ClockSampler.FIELDS, restricted to samples taken in [t_begin, t_end + slack]."""
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    parsed = []
    for t, ln in lines:
        parts = [x.strip() for x in ln.split(",")]
        if len(parts) < 8:
            continue
        try:
            sm, mx = float(parts[1]), float(parts[2])
        except ValueError:
            continue
        parsed.append((_sample_time(parts[0], t), sm, mx,
                       [nm for nm, v in zip(names, parts[4:8]) if v.lower() == "active"]))
    window = parsed
    in_region = True
    if t_begin is not None and t_end is not None:
        window = [p for p in parsed if t_begin <= p[0] <= t_end + slack]
        if not window:
            window, in_region = parsed, False
    reasons = sorted({r for p in window for r in p[3]})
    out = {"sm_mhz": float(np.median([p[1] for p in window])) if window else None,
           "sm_max_mhz": max(p[2] for p in window) if window else None,
           "reasons": reasons, "samples": len(window)}
    if not in_region:
        out["note"] = "no sample inside the timed region; all samples of the run are summarised"
    return out


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def reduce_over_ranks(dist, ms, tokens, device):
    """Whole-job timing of N replicas: the slowest rank's time and the
    tokens of all ranks."""
    import torch
    t = torch.tensor([ms, tokens], dtype=torch.float64, device=device)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    total = t.clone()
    dist.all_reduce(total, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(total[1])


def build_model(args, torch):
    import synth
    import speculative_decoding_verify_pass_gb300 as sv
    cfg = synth.PRESETS[args.config](max_ctx=args.ctx + 1024)
    if args.layers:
        cfg = synth.scaled(cfg, n_layers=args.layers)
    t0 = time.time()
    w = synth.make_weights(cfg)
    t_gen = time.time() - t0
    plan = sv.layer_skip_plan(cfg.n_layers, args.skip)
    m = sv.Model(cfg, w, draft_plan=plan)
    return cfg, w, plan, m, t_gen


def load_synthetic_context(m, cfg, plan, ctx):
    """Fill both caches with the seeded N(0,1) keys/values of positions
    0..ctx-1 (the same context the oracle arm uses)."""
    import synth
    for l in range(cfg.n_layers):
        k = synth.synthetic_kv(cfg, l, ctx, 0)
        v = synth.synthetic_kv(cfg, l, ctx, 1)
        m.kv_load(0, l, k, v)
        if l in plan:
            m.kv_load(1, plan.index(l), k, v)


def device_cycles(m, torch, gamma, steps, buf, acc_log, start_idx):
    """`steps` device-resident cycles.  buf[0] = token at the last kept
    position, buf[1] = last accepted token, buf[2..] = drafts."""
    import speculative_decoding_verify_pass_gb300 as sv
    launches = 0
    n = gamma + 1
    am = torch.zeros(n, dtype=torch.int32, device="cuda")
    for s in range(steps):
        sv.spec_draft_step(m.h, buf[0:2], buf[2:3])
        launches += m.launches()
        for i in range(1, gamma):
            sv.spec_draft_step(m.h, buf[1 + i:2 + i], buf[2 + i:3 + i])
            launches += m.launches()
        sv.spec_verify_step(m.h, buf[1:1 + n], am, acc_log[start_idx + s:start_idx + s + 1], None, None, buf[0:2])
        launches += m.launches()
        sv.spec_kv_rollback(m.h, sv.SPEC_CACHE_TARGET, -1)
        launches += m.launches()
        sv.spec_kv_rollback(m.h, sv.SPEC_CACHE_DRAFT, -1)
        launches += m.launches()
    return launches


# ----------------------------------------------------------------------------
# Default workload: verify cycles with geometric acceptance (Llama-3.1-8B shape)
# ----------------------------------------------------------------------------
def geometric_schedule(n, alpha, count, vocab):
    """(block start, accept length) of `count` verify cycles of n tokens whose
    n-1 drafts come from synth.corrupt_drafts (stream = cycle index).  Which
    drafts stay clean depends only on the seeded stream, not on the tokens,
    so the accept length (the number of leading clean drafts) of every cycle,
    and with it where the next block starts, is known before the run."""
    import synth
    j, out = 0, []
    for s in range(count):
        k = 0
        if n > 1:
            dummy = np.zeros(n - 1, dtype=np.int32)
            clean = synth.corrupt_drafts(dummy, alpha, vocab, stream=s) == dummy
            while k < n - 1 and clean[k]:
                k += 1
        out.append((j, k))
        j += k + 1
    return out


def geometric_blocks(greedy, sched, n, alpha, vocab):
    """Blocks [greedy[j]] + corrupt_drafts(greedy[j+1 .. j+n-1]) of the
    schedule; checks that each accepts exactly its scheduled length."""
    import synth
    blocks = np.zeros((len(sched), n), dtype=np.int32)
    for s, (j, k) in enumerate(sched):
        truth = np.array(greedy[j + 1:j + n], dtype=np.int32)
        drafts = synth.corrupt_drafts(truth, alpha, vocab, stream=s) if n > 1 else truth
        blocks[s, 0] = greedy[j]
        blocks[s, 1:] = drafts
        lead = 0
        while lead < n - 1 and drafts[lead] == truth[lead]:
            lead += 1
        assert lead == k, (s, lead, k)
    return blocks


def launch_segments(stamps, kinds):
    """Split one traced pass ([ctas][launches][entry, ready, work, exit]
    global-timer stamps) into consecutive per-launch segments: launch i owns
    the time from the previous launch's last CTA exit (or its own first
    entry, for the first launch) to its own last CTA exit.  The segments
    tile the pass, so their sum over any set of launches is at most the pass
    time.  Returns [(kind, microseconds)] in launch order."""
    out, prev = [], None
    for l, kind in enumerate(kinds):
        s = stamps[:, l, :]
        live = s[s[:, 0] > 0]
        if len(live) == 0:
            continue
        ex = int(live[:, 3].max())
        start = int(live[:, 0].min()) if prev is None else prev
        out.append((int(kind), max(ex - start, 0) / 1e3))
        prev = ex if prev is None else max(prev, ex)
    return out


GEMM_KINDS = (0, 1, 2, 3)      # QKV, residual (O / down), SwiGLU gate-up, LM head


def inpipeline_gemm_roofline(m, torch, sv, blk, ctx, peak, peak_kind, cfg, args, reps=3):
    """The streaming GEMM inside an unbracketed verify pass: algorithmic bytes
    per pass (from one event-profiled pass) over the GEMM launches' trace
    segments (launch_segments), averaged over `reps` traced passes."""
    n = blk.numel()
    am = torch.zeros(n, dtype=torch.int32, device="cuda")
    ac = torch.zeros(1, dtype=torch.int32, device="cuda")
    sv.spec_profile_enable(m.h, True)
    sv.spec_verify_step(m.h, blk, am, ac)
    sv.spec_kv_rollback(m.h, 0, ctx)
    per_kind = {k: sv.spec_profile_read(m.h, k) for k in GEMM_KINDS}
    sv.spec_profile_enable(m.h, False)
    traffic, traffic_note = ncu_traffic({k: v[2] for k, v in per_kind.items()}, cfg, args)
    gbytes = sum(v[1] for v in per_kind.values())
    glaunch = sum(v[2] for v in per_kind.values())
    sv.spec_trace_enable(m.h, True)
    seg_us, span_us = [], []
    for r in range(reps + 1):
        sv.spec_verify_step(m.h, blk, am, ac)
        sv.spec_kv_rollback(m.h, 0, ctx)
        torch.cuda.synchronize()
        if r == 0:
            continue     # the first traced pass warms the direct-launch path
        segs = launch_segments(sv.spec_trace_read(m.h), sv.spec_trace_kinds(m.h))
        seg_us.append(sum(t for k, t in segs if k in GEMM_KINDS))
        span_us.append(sum(t for _, t in segs))
    sv.spec_trace_enable(m.h, False)
    gus = float(np.mean(seg_us))
    achieved = gbytes / (gus * 1e-6) / 1e9
    return {"kernel": "gemm_kernel (weight-streaming GEMM: QKV, O, gate-up, down, LM head)", "bound": "hbm",
            "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic, "traffic_source": traffic_note,
            "timing": "global-timer launch trace of unbracketed verify passes: each launch owns the time from the "
                      "previous launch's last CTA exit to its own last CTA exit, so the GEMM segments plus the "
                      "other launches' segments add up to the traced pass",
            "launches_per_pass": glaunch, "bytes_per_launch": round(gbytes / max(glaunch, 1)),
            "avg_launch_us": round(gus / max(glaunch, 1), 2), "gemm_us_per_pass": round(gus, 1),
            "traced_pass_us": round(float(np.mean(span_us)), 1)}


def run_native(args):
    if args.workload == "selfspec":
        return run_native_selfspec(args)
    return run_native_geometric(args)


def run_native_geometric(args):
    import torch
    import speculative_decoding_verify_pass_gb300 as sv
    import synth
    from speculative_decoding_verify_pass_gb300 import stepmodel

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import __graft_entry__
    __graft_entry__.build()

    n, alpha, ctx = args.n, args.alpha, args.ctx
    total = args.warmup + args.steps
    sched = geometric_schedule(n, alpha, total, synth.PRESETS[args.config]().vocab)
    span = sched[-1][0] + n + 1                        # positions the cycles advance through
    cfg = synth.PRESETS[args.config](max_ctx=ctx + span + 64)
    if args.layers:
        cfg = synth.scaled(cfg, n_layers=args.layers)
    t0 = time.time()
    w = synth.make_weights(cfg)
    t_gen = time.time() - t0
    m = sv.Model(cfg, w)
    load_synthetic_context(m, cfg, [], ctx)
    m.kv_set_len(sv.SPEC_CACHE_TARGET, ctx)
    m.check_error()
    # the target's own greedy continuation of the context (verify passes of one token)
    y0 = int(synth.prompt(cfg, 1)[0])
    greedy = [y0]
    one = torch.zeros(1, dtype=torch.int32, device="cuda")
    am1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    ac1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    while len(greedy) < span:
        one.fill_(greedy[-1])
        sv.spec_verify_step(m.h, one, am1, ac1)
        greedy.append(int(am1.item()))
    sv.spec_kv_rollback(m.h, sv.SPEC_CACHE_TARGET, ctx)
    blocks = geometric_blocks(greedy, sched, n, alpha, cfg.vocab)
    d_blocks = torch.from_numpy(blocks).to("cuda")
    blk = torch.zeros(n, dtype=torch.int32, device="cuda")
    am = torch.zeros(n, dtype=torch.int32, device="cuda")
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    acc_log = torch.zeros(total, dtype=torch.int32, device="cuda")

    def cycles(s0, count):
        launches = 0
        for s in range(s0, s0 + count):
            blk.copy_(d_blocks[s])
            sv.spec_verify_step(m.h, blk, am, acc)
            launches += m.launches()
            acc_log[s:s + 1].copy_(acc)
            sv.spec_kv_rollback(m.h, sv.SPEC_CACHE_TARGET, -1)
            launches += m.launches()
        return launches

    cycles(0, args.warmup)
    torch.cuda.synchronize()
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        uuid = None
    clk = ClockSampler(uuid)
    clk.start()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_begin = time.time()
    e0.record(stream)
    torch.cuda.nvtx.range_push("timed")      # lets a launch-list capture select exactly these launches
    launches = cycles(args.warmup, args.steps)
    torch.cuda.nvtx.range_pop()
    e1.record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    if dist:
        dist.barrier()
    clocks = clk.stop(t_begin, t_end)
    ms = e0.elapsed_time(e1)
    m.check_error()
    got = acc_log.cpu().numpy()
    want = np.array([k for _, k in sched], dtype=np.int32)
    schedule_ok = bool(np.array_equal(got, want))
    timed = got[args.warmup:total]
    tokens = float(np.sum(timed + 1))
    ctx_end = m.kv_len(sv.SPEC_CACHE_TARGET)
    step_bytes = float(np.mean([pass_bytes(cfg, n, ctx + j) for j, _ in sched[args.warmup:total]]))
    if dist:
        ms, tokens = reduce_over_ranks(dist, ms, tokens, "cuda")
    value = tokens / (ms / 1e3)
    us_step = ms * 1e3 / args.steps
    peak, peak_kind = measured_peaks()

    # ---- verify pass alone, per block size, at context ctx ----
    sweep = {}
    for nn in range(1, n + 1):
        us = _verify_us(torch, sv, m, [int(t) for t in blocks[0, :nn]], ctx)
        b = pass_bytes(cfg, nn, ctx)
        e_tok = stepmodel.tokens_per_verify(alpha, nn - 1)
        sweep[str(nn)] = {"us": round(us, 1), "GBps": round(b / us / 1e3, 1),
                          "frac_8TBps": round(b / us / 1e3 / NOMINAL_HBM, 3),
                          "frac_measured_peak": round(b / us / 1e3 / peak, 3),
                          "expected_tokens": round(e_tok, 3), "expected_tok_s": round(e_tok / us * 1e6, 1)}

    # ---- dominant kernel: the streaming GEMM inside unbracketed passes ----
    blk.copy_(d_blocks[0])
    roof = inpipeline_gemm_roofline(m, torch, sv, blk, ctx, peak, peak_kind, cfg, args)

    # ---- end to end through the host-driven API (pinned copies each step) ----
    e2e = run_e2e_geometric(m, torch, sv, blocks, sched, ctx, args)

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "%s verify cycles at KV context %d (seeded synthetic KV), block n=%d (last accepted "
                               "token + %d drafts), drafts = seeded corruptions of the target's greedy tokens with "
                               "geometric acceptance alpha=%.2f; verify + accept + device rollback per step" % (
                                   cfg.name, ctx, n, n - 1, alpha),
                   "model": cfg.name + "-shaped, random-init N(0,0.02) bf16" + (
                       ", first %d layers only" % args.layers if args.layers else ""),
                   "global_batch": world, "seq_len": ctx, "n": n, "alpha": alpha,
                   "context_range": [ctx + sched[args.warmup][0], ctx_end],
                   "l2": "no flush: %.1f GB of weights and KV per step exceed the 129 MB L2" % (step_bytes / 1e9),
                   "parallelism": "replicas" if world > 1 else "single"},
        "accept_mean": round(float(np.mean(timed)), 4),
        "accept_schedule_matched": schedule_ok,
        "verify": {"n": n, "us_per_step": round(us_step, 1), "bytes_per_step": round(step_bytes),
                   "GBps": round(step_bytes / us_step / 1e3, 1),
                   "frac_8TBps": round(step_bytes / us_step / 1e3 / NOMINAL_HBM, 3),
                   "frac_measured_peak": round(step_bytes / us_step / 1e3 / peak, 3), "by_n": sweep},
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "weights_gen_s": round(t_gen, 1),
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline_geometric(cfg, w, sched, args)
    m.close()
    if dist:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


def run_e2e_geometric(m, torch, sv, blocks, sched, ctx, args):
    """The same cycles driven from the host: each step copies its block from
    pinned host memory to the device, runs the verify, reads the argmax rows
    and accept_len back into pinned memory, and rolls the cache back with
    the host's exact length."""
    n = blocks.shape[1]
    pin_in = torch.zeros(n, dtype=torch.int32).pin_memory()
    pin_out = torch.zeros(n + 1, dtype=torch.int32).pin_memory()
    dev_in = torch.zeros(n, dtype=torch.int32, device="cuda")
    am = torch.zeros(n, dtype=torch.int32, device="cuda")
    out = torch.zeros(n + 1, dtype=torch.int32, device="cuda")
    steps = min(max(3, args.steps), len(sched))
    host_blocks = torch.from_numpy(blocks)
    pos = ctx
    sv.spec_kv_rollback(m.h, 0, pos)
    tokens, matched = 0, True
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(steps):
        pin_in.copy_(host_blocks[s])
        dev_in.copy_(pin_in, non_blocking=True)
        sv.spec_verify_step(m.h, dev_in, am, out[n:n + 1])
        out[:n].copy_(am)
        pin_out.copy_(out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        k = int(pin_out[n])
        matched = matched and k == sched[s][1]
        sv.spec_kv_rollback(m.h, 0, pos + k + 1)
        pos += k + 1
        tokens += k + 1
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    return {"value": round(tokens / dt, 2), "unit": "tok/s", "h2d_bytes_per_step": 4 * n,
            "d2h_bytes_per_step": 4 * (n + 1), "steps": steps, "accept_schedule_matched": matched}


def oracle_verify_setup(cfg, w, ctx):
    import oracle
    import synth
    orc = oracle.Oracle(cfg, w)
    tc = orc.new_cache()
    for l in range(cfg.n_layers):
        tc.load(l, synth.synthetic_kv(cfg, l, ctx, 0).reshape(ctx, -1),
                synth.synthetic_kv(cfg, l, ctx, 1).reshape(ctx, -1))
    tc.set_len(ctx)
    return orc, tc


def cpu_baseline_geometric(cfg, w, sched, args, min_seconds=10.0, max_passes=30):
    """The oracle on the host cores: verify passes of n tokens at context ctx
    (the block's token ids from synth.prompt; the time does not depend on
    them), each credited with the tokens its cycle of the acceptance
    schedule emits, repeated until about min_seconds of CPU work."""
    import oracle
    import synth
    orc, tc = oracle_verify_setup(cfg, w, args.ctx)
    block = [int(t) for t in synth.prompt(cfg, args.n, stream=5)]
    t0 = time.perf_counter()
    toks, passes = 0, 0
    while passes < max_passes and (passes == 0 or time.perf_counter() - t0 < min_seconds):
        orc.forward(tc, orc.full_plan, block, args.ctx)
        tc.truncate(args.ctx)
        toks += sched[passes % len(sched)][1] + 1
        passes += 1
    dt = time.perf_counter() - t0
    cores = oracle.get_threads()
    return {"value": round(toks / dt, 4), "unit": "tok/s", "cores": cores, "kind": "oracle",
            "sample": "%d verify passes (n=%d, all %d layers, context %d, synthetic seeded KV) of the fp32 C oracle, "
                      "%.1f s; tokens per pass from the same acceptance schedule as the GPU arm" % (
                          passes, args.n, cfg.n_layers, args.ctx, dt),
            "verify_pass_ms": oracle_verify_ms(orc, tc, args.n, args.ctx, block, cores)}


def run_reference_geometric(args):
    import oracle
    import synth
    oracle.build()
    synth.build()
    total = args.warmup + args.steps
    sched = geometric_schedule(args.n, args.alpha, total, synth.PRESETS[args.config]().vocab)
    cfg = synth.PRESETS[args.config](max_ctx=args.ctx + 64)
    if args.layers:
        cfg = synth.scaled(cfg, n_layers=args.layers)
    w = synth.make_weights(cfg)
    orc, tc = oracle_verify_setup(cfg, w, args.ctx)
    block = [int(t) for t in synth.prompt(cfg, args.n, stream=5)]
    for _ in range(args.warmup):
        orc.forward(tc, orc.full_plan, block, args.ctx)
        tc.truncate(args.ctx)
    t0 = time.perf_counter()
    toks = 0
    for s in range(args.warmup, total):
        orc.forward(tc, orc.full_plan, block, args.ctx)
        tc.truncate(args.ctx)
        toks += sched[s][1] + 1
    dt = time.perf_counter() - t0
    value = toks / dt
    sample = ("each step one verify pass (n=%d, all %d layers) of the fp32 C oracle at context %d on synthetic seeded "
              "KV, credited with the tokens of the same geometric acceptance schedule (alpha=%.2f) as the GPU arm" % (
                  args.n, cfg.n_layers, args.ctx, args.alpha))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tok/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "%s verify cycles at KV context %d, block n=%d, geometric acceptance alpha=%.2f" % (
            cfg.name, args.ctx, args.n, args.alpha), "seq_len": args.ctx, "n": args.n, "alpha": args.alpha},
        "cpu_baseline": {"value": round(value, 4), "unit": "tok/s", "cores": oracle.get_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


def run_native_selfspec(args):
    import torch
    import speculative_decoding_verify_pass_gb300 as sv
    import synth

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import __graft_entry__
    __graft_entry__.build()

    cfg, w, plan, m, t_gen = build_model(args, torch)
    gamma, ctx = args.gamma, args.ctx
    n = gamma + 1
    prompt = synth.prompt(cfg, ctx)
    load_synthetic_context(m, cfg, plan, ctx)
    m.check_error()
    # device loop state: draft cache one behind the target for the catch-up pair
    buf = torch.zeros(2 + gamma, dtype=torch.int32, device="cuda")
    buf[0] = int(prompt[-2])
    buf[1] = int(prompt[-1])
    m.kv_set_len(sv.SPEC_CACHE_TARGET, ctx)
    m.kv_set_len(sv.SPEC_CACHE_DRAFT, ctx - 1)
    total = args.warmup + args.steps
    acc_log = torch.zeros(total + 1, dtype=torch.int32, device="cuda")
    device_cycles(m, torch, gamma, args.warmup, buf, acc_log, 0)
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        uuid = None
    clk = ClockSampler(uuid)
    clk.start()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_begin = time.time()
    e0.record(stream)
    torch.cuda.nvtx.range_push("timed")      # lets a launch-list capture select exactly these launches
    launches = device_cycles(m, torch, gamma, args.steps, buf, acc_log, args.warmup)
    torch.cuda.nvtx.range_pop()
    e1.record(stream)
    torch.cuda.synchronize()
    t_end = time.time()
    if dist:
        dist.barrier()
    clocks = clk.stop(t_begin, t_end)
    ms = e0.elapsed_time(e1)
    m.check_error()
    accepts = acc_log[args.warmup:total].cpu().numpy()
    tokens = float(np.sum(accepts + 1))
    if dist:
        ms, tokens = reduce_over_ranks(dist, ms, tokens, "cuda")
    value = tokens / (ms / 1e3)
    ctx_now = m.kv_len(sv.SPEC_CACHE_TARGET)

    # ---- verify pass alone, per block size (context held at ctx_now) ----
    sweep = {}
    for nn in sorted(set([1, 2, 3, 4, 6, 8, 16, n])):
        blk = torch.tensor(prompt[:nn], dtype=torch.int32, device="cuda")
        am = torch.zeros(nn, dtype=torch.int32, device="cuda")
        ac = torch.zeros(1, dtype=torch.int32, device="cuda")
        for _ in range(3):
            sv.spec_verify_step(m.h, blk, am, ac)
            sv.spec_kv_rollback(m.h, 0, ctx_now)
        reps = 10
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(reps):
            sv.spec_verify_step(m.h, blk, am, ac)
            sv.spec_kv_rollback(m.h, 0, ctx_now)
        a1.record(stream)
        torch.cuda.synchronize()
        us = a0.elapsed_time(a1) * 1e3 / reps
        b = pass_bytes(cfg, nn, ctx_now)
        sweep[str(nn)] = {"us": round(us, 1), "GBps": round(b / us / 1e3, 1),
                          "frac_8TBps": round(b / us / 1e3 / NOMINAL_HBM, 3)}

    # ---- dominant kernel: the streaming GEMM, events around each launch ----
    sv.spec_profile_enable(m.h, True)
    device_cycles(m, torch, gamma, 3, buf, acc_log, total - 3)
    per_kind = {k: sv.spec_profile_read(m.h, k) for k in (sv.EPI_QKV, sv.EPI_RESID, sv.EPI_SWIGLU, sv.EPI_LMHEAD)}
    sv.spec_profile_enable(m.h, False)
    gms = sum(v[0] for v in per_kind.values())
    gbytes = sum(v[1] for v in per_kind.values())
    glaunch = sum(v[2] for v in per_kind.values())
    peak, peak_kind = measured_peaks()
    achieved = gbytes / (gms / 1e3) / 1e9 if gms > 0 else 0.0
    traffic, traffic_note = ncu_traffic({k: v[2] for k, v in per_kind.items()}, cfg, args)

    # ---- end to end through the host-driven API (pinned copies each step) ----
    e2e = run_e2e(m, torch, sv, gamma, args, prompt, ctx_now)

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "%s self-speculative cycle at context %d (seeded synthetic KV): %d draft steps over the "
                               "%d%% middle-skip plan (%d of %d layers) + verify n=%d + accept + rollback" % (
                                   cfg.name, ctx, gamma, round(args.skip * 100), len(plan), cfg.n_layers, n),
                   "model": cfg.name + "-shaped, random-init N(0,0.02) bf16" + (
                       ", first %d layers only" % args.layers if args.layers else ""),
                   "global_batch": world, "seq_len": ctx,
                   "gamma": gamma, "skip_frac": args.skip, "draft_layers": len(plan),
                   "l2": "no flush: %.1f GB of weights per cycle exceed the 129 MB L2" % (pass_bytes(cfg, n, ctx) / 1e9),
                   "parallelism": "replicas" if world > 1 else "single"},
        "accept_mean": round(float(np.mean(accepts)), 4),
        "verify": {"n": n, "us": sweep[str(n)]["us"], "GBps": sweep[str(n)]["GBps"],
                   "frac_8TBps": sweep[str(n)]["frac_8TBps"],
                   "frac_measured_peak": round(sweep[str(n)]["GBps"] / peak, 3), "bytes": pass_bytes(cfg, n, ctx_now),
                   "by_n": sweep},
        "roofline": {"kernel": "gemm_kernel (weight-streaming GEMM, all dense epilogues)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "traffic_source": traffic_note,
                     "launches_timed": glaunch, "bytes_per_launch": round(gbytes / max(glaunch, 1)),
                     "avg_launch_us": round(gms * 1e3 / max(glaunch, 1), 2)},
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
        "weights_gen_s": round(t_gen, 1),
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(cfg, w, plan, args, prompt)
    m.close()
    if dist:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


def run_e2e(m, torch, sv, gamma, args, prompt, ctx_now):
    """Host-driven cycles: each step copies its input tokens from pinned host
    memory, runs the cycle through the public calls and reads the argmax rows
    and accept_len back (host rollback with exact values)."""
    n = gamma + 1
    pin_in = torch.zeros(2, dtype=torch.int32).pin_memory()
    pin_out = torch.zeros(n + 1, dtype=torch.int32).pin_memory()
    dev_in = torch.zeros(2, dtype=torch.int32, device="cuda")
    drafts = torch.zeros(gamma + 1, dtype=torch.int32, device="cuda")
    am = torch.zeros(n, dtype=torch.int32, device="cuda")
    out = torch.zeros(n + 1, dtype=torch.int32, device="cuda")
    pos = ctx_now           # target length; the last accepted token goes to this position
    sv.spec_kv_rollback(m.h, 0, pos)
    sv.spec_kv_rollback(m.h, 1, pos - 1)
    prev, last = int(prompt[-1]), int(prompt[-2])
    tokens = 0
    steps = max(3, args.steps)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(steps):
        pin_in[0] = prev
        pin_in[1] = last
        dev_in.copy_(pin_in, non_blocking=True)
        sv.spec_draft_step(m.h, dev_in, drafts[1:2])
        for i in range(1, gamma):
            sv.spec_draft_step(m.h, drafts[i:i + 1], drafts[i + 1:i + 2])
        drafts[0:1].copy_(dev_in[1:2])
        sv.spec_verify_step(m.h, drafts[0:n], am, out[n:n + 1])
        out[:n].copy_(am)
        pin_out.copy_(out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        k = int(pin_out[n])
        a = pin_out[:n].tolist()
        prev = last if k == 0 else int(drafts[k].item())
        new_last = a[k]
        tokens += k + 1
        sv.spec_kv_rollback(m.h, 0, pos + k + 1)
        sv.spec_kv_rollback(m.h, 1, pos + k)
        pos = pos + k + 1
        last = new_last
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    return {"value": round(tokens / dt, 2), "unit": "tok/s", "h2d_bytes_per_step": 8,
            "d2h_bytes_per_step": 4 * (n + 1), "steps": steps}


# ----------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ----------------------------------------------------------------------------
def oracle_cycle_setup(cfg, w, plan, ctx):
    import oracle
    import synth
    orc = oracle.Oracle(cfg, w)
    tc = orc.new_cache()
    dc = orc.new_cache(len(plan))
    for l in range(cfg.n_layers):
        k = synth.synthetic_kv(cfg, l, ctx, 0).reshape(ctx, -1)
        v = synth.synthetic_kv(cfg, l, ctx, 1).reshape(ctx, -1)
        tc.load(l, k, v)
        if l in plan:
            dc.load(plan.index(l), k, v)
    tc.set_len(ctx)
    dc.set_len(ctx)
    return orc, tc, dc


def oracle_cycle(orc, tc, dc, plan, gamma, ctx, y):
    """One cycle on the oracle at context ctx (then cropped back to ctx)."""
    import oracle
    feed = [y]
    drafts = []
    for _ in range(gamma):
        lg, _, _ = orc.forward(dc, plan, feed, dc.len, logits_from=len(feed) - 1)
        drafts.append(oracle.argmax(lg[-1]))
        feed = [drafts[-1]]
    block = [y] + drafts
    lg, _, _ = orc.forward(tc, orc.full_plan, block, ctx)
    a = [oracle.argmax(r) for r in lg]
    k = oracle.accept_len(block, a)
    tc.truncate(ctx)
    dc.truncate(ctx)
    return k + 1


def cpu_baseline(cfg, w, plan, args, prompt, min_seconds=10.0, max_cycles=30):
    """The oracle on the host cores: whole cycles of the bench's workload,
    repeated until about min_seconds of CPU work (a bounded sample)."""
    import oracle
    orc, tc, dc = oracle_cycle_setup(cfg, w, plan, args.ctx)
    t0 = time.perf_counter()
    toks, cycles = 0, 0
    while cycles < max_cycles and (cycles == 0 or time.perf_counter() - t0 < min_seconds):
        toks += oracle_cycle(orc, tc, dc, plan, args.gamma, args.ctx, int(prompt[-1]))
        cycles += 1
    dt = time.perf_counter() - t0
    cores = oracle.get_threads()
    return {"value": round(toks / dt, 4), "unit": "tok/s", "cores": cores, "kind": "oracle",
            "sample": "%d cycles (each %d draft passes + verify n=%d) at context %d on synthetic seeded KV, "
                      "fp32 C oracle, %.1f s" % (cycles, args.gamma, args.gamma + 1, args.ctx, dt),
            "verify_pass_ms": oracle_verify_ms(orc, tc, args.gamma + 1, args.ctx, prompt, cores)}


def oracle_verify_ms(orc, tc, n, ctx, prompt, cores):
    """One verify pass of n tokens at context ctx on the oracle, wall clock,
    on all the host's cores and on one core."""
    import oracle
    block = [int(t) for t in prompt[:n]]
    out = {}
    for label, threads in (("all_cores", cores), ("one_core", 1)):
        oracle.set_threads(threads)
        t0 = time.perf_counter()
        orc.forward(tc, orc.full_plan, block, ctx)
        out[label] = round((time.perf_counter() - t0) * 1e3, 1)
        tc.truncate(ctx)
    oracle.set_threads(cores)
    out["cores"] = cores
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    if args.workload != "selfspec":
        return run_reference_geometric(args)
    import oracle
    import synth
    oracle.build()
    synth.build()
    cfg = synth.PRESETS[args.config](max_ctx=args.ctx + 64)
    w = synth.make_weights(cfg)
    plan = oracle.layer_skip_plan(cfg.n_layers, args.skip)
    orc, tc, dc = oracle_cycle_setup(cfg, w, plan, args.ctx)
    prompt = synth.prompt(cfg, args.ctx)
    y = int(prompt[-1])
    for _ in range(args.warmup):
        oracle_cycle(orc, tc, dc, plan, args.gamma, args.ctx, y)
    t0 = time.perf_counter()
    toks = 0
    for _ in range(args.steps):
        toks += oracle_cycle(orc, tc, dc, plan, args.gamma, args.ctx, y)
    dt = time.perf_counter() - t0
    value = toks / dt
    n = args.gamma + 1
    sample = ("each step one full cycle (%d draft passes + verify n=%d) of the fp32 C oracle at context %d on "
              "synthetic seeded KV" % (args.gamma, n, args.ctx))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tok/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "%s self-speculative cycle at context %d, gamma %d, %d%% middle skip" % (
            cfg.name, args.ctx, args.gamma, round(args.skip * 100)), "seq_len": args.ctx, "gamma": args.gamma},
        "cpu_baseline": {"value": round(value, 4), "unit": "tok/s", "cores": oracle.get_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))


# ----------------------------------------------------------------------------
# measurement suites (one JSON line per point; not the default bench line)
# ----------------------------------------------------------------------------
def _emit(d):
    print(json.dumps(d), flush=True)


def _model_at_context(cfg, ctx, draft_plan=None):
    import synth
    import speculative_decoding_verify_pass_gb300 as sv
    w = synth.make_weights(cfg)
    m = sv.Model(cfg, w, draft_plan=draft_plan)
    plan = draft_plan or []
    for l in range(cfg.n_layers):
        k = synth.synthetic_kv(cfg, l, ctx, 0)
        v = synth.synthetic_kv(cfg, l, ctx, 1)
        m.kv_load(0, l, k, v)
        if l in plan:
            m.kv_load(1, plan.index(l), k, v)
    m.kv_set_len(0, ctx)
    if plan:
        m.kv_set_len(1, ctx)
    return m, w


def _time_calls(torch, fn, reps=10, warm=3):
    for _ in range(warm):
        fn()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / reps  # us


def _verify_us(torch, sv, m, toks, ctx, reps=10):
    n = len(toks)
    blk = torch.tensor(toks, dtype=torch.int32, device="cuda")
    am = torch.zeros(n, dtype=torch.int32, device="cuda")
    ac = torch.zeros(1, dtype=torch.int32, device="cuda")

    def one():
        sv.spec_verify_step(m.h, blk, am, ac)
        sv.spec_kv_rollback(m.h, 0, ctx)
    return _time_calls(torch, one, reps)


def _draft_us(torch, sv, m, ctx, reps=10):
    t = torch.tensor([1], dtype=torch.int32, device="cuda")
    out = torch.zeros(1, dtype=torch.int32, device="cuda")

    def one():
        sv.spec_draft_step(m.h, t, out)
        sv.spec_kv_rollback(m.h, 1, ctx)
    return _time_calls(torch, one, reps)


def suite_sweep(args):
    """Verify time / HBM bandwidth vs block size, and draft-step time vs skip
    fraction (the MLX post's sweep), for the dense workload shapes."""
    import torch
    import synth
    import speculative_decoding_verify_pass_gb300 as sv
    from speculative_decoding_verify_pass_gb300 import stepmodel
    peak, _ = measured_peaks()
    jobs = [("qwen3-4b", 2048, (1, 2, 3, 4, 6, 8, 12, 16)), ("llama-3.1-8b", 4096, (1, 2, 4, 8, 16)),
            ("qwen3-8b", 1024, (1, 16)), ("qwen3-8b", 2048, (1, 16)), ("qwen3-8b", 4096, (1, 4, 16))]
    for name, ctx, ns in jobs:
        cfg = synth.PRESETS[name](max_ctx=ctx + 64)
        plan = sv.layer_skip_plan(cfg.n_layers, 0.5)
        m, _ = _model_at_context(cfg, ctx, plan)
        for n in ns:
            us = _verify_us(torch, sv, m, synth.prompt(cfg, n).tolist(), ctx)
            b = stepmodel.pass_bytes(cfg, n, ctx)
            _emit({"suite": "verify", "config": name, "ctx": ctx, "n": n, "us": round(us, 1),
                   "GBps": round(b / us / 1e3, 1), "frac_8TBps": round(b / us / 1e3 / NOMINAL_HBM, 3),
                   "frac_measured": round(b / us / 1e3 / peak, 3)})
        if name != "qwen3-8b" or ctx == 2048:
            for f in (0.1, 0.2, 0.3, 0.4, 0.5):
                plan = sv.layer_skip_plan(cfg.n_layers, f)
                m.set_draft_plan(plan)
                import numpy as np
                for l in plan:
                    m.kv_load(1, plan.index(l), synth.synthetic_kv(cfg, l, ctx, 0), synth.synthetic_kv(cfg, l, ctx, 1))
                m.kv_set_len(1, ctx)
                us = _draft_us(torch, sv, m, ctx)
                b = stepmodel.pass_bytes(cfg, 1, ctx, plan)
                _emit({"suite": "draft", "config": name, "ctx": ctx, "skip_frac": f, "layers": len(plan),
                       "us": round(us, 1), "GBps": round(b / us / 1e3, 1)})
        m.close()
        del m
        torch.cuda.empty_cache()


def suite_geometric(args):
    """Llama-3.1-8B verify at n = 1..8 with drafts that are seeded corruptions
    of the target's own greedy tokens (acceptance geometric in alpha); the
    accepted tokens per second of the verify loop."""
    import numpy as np
    import torch
    import synth
    import speculative_decoding_verify_pass_gb300 as sv
    from speculative_decoding_verify_pass_gb300 import stepmodel
    ctx = 4096
    cfg = synth.llama31_8b(max_ctx=ctx + 256)
    m, _ = _model_at_context(cfg, ctx)
    # the target's own greedy continuation from the context
    y = int(synth.prompt(cfg, 1)[0])
    greedy = [y]
    blk = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(96):
        blk.fill_(greedy[-1])
        am, _, _, _ = m.verify(blk)
        greedy.append(int(am.item()))
    for alpha in (0.5, 0.7, 0.9):
        for n in range(1, 9):
            m.kv_set_len(0, ctx)
            pos, toks, cyc = 0, 0, 0
            am = torch.zeros(n, dtype=torch.int32, device="cuda")
            ac = torch.zeros(1, dtype=torch.int32, device="cuda")
            accepts = []
            t_total = 0.0
            while pos + n < len(greedy) and cyc < 24:
                truth = greedy[pos + 1:pos + n]
                drafts = synth.corrupt_drafts(np.array(truth, dtype=np.int32), alpha, cfg.vocab,
                                              stream=1000 * n + cyc).tolist() if n > 1 else []
                b = torch.tensor([greedy[pos]] + drafts, dtype=torch.int32, device="cuda")
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                sv.spec_verify_step(m.h, b, am, ac)
                sv.spec_kv_rollback(m.h, 0, -1)
                e1.record()
                torch.cuda.synchronize()
                k = int(ac.item())
                t_total += e0.elapsed_time(e1) * 1e-3
                accepts.append(k)
                toks += k + 1
                pos += k + 1
                cyc += 1
            _emit({"suite": "geometric", "config": "llama-3.1-8b", "ctx": ctx, "alpha": alpha, "n": n,
                   "cycles": cyc, "accept_mean": round(float(np.mean(accepts)), 3),
                   "expected_tokens": round(stepmodel.tokens_per_verify(alpha, n - 1), 3),
                   "tokens_per_cycle": round(toks / max(cyc, 1), 3), "us_per_verify": round(t_total / cyc * 1e6, 1),
                   "accepted_tok_s": round(toks / t_total, 1)})
    m.close()


DFLASH_TAP_LAYERS = [1, 9, 17, 25, 33]


def suite_dflash(args):
    """Qwen3-8B verify of a 16-token block (the DFlash block size) at context
    1024/2048/4096, accept lengths truncated-geometric with mean 6 and 9, then
    the rollback of the rejected tail."""
    import numpy as np
    import torch
    import synth
    import speculative_decoding_verify_pass_gb300 as sv
    from speculative_decoding_verify_pass_gb300 import stepmodel
    for ctx in (1024, 2048, 4096):
        cfg = synth.qwen3_8b(max_ctx=ctx + 64)
        m, _ = _model_at_context(cfg, ctx)
        blk = torch.tensor(synth.prompt(cfg, 16).tolist(), dtype=torch.int32, device="cuda")
        am = torch.zeros(16, dtype=torch.int32, device="cuda")
        ac = torch.zeros(1, dtype=torch.int32, device="cuda")
        us_v = _time_calls(torch, lambda: (sv.spec_verify_step(m.h, blk, am, ac), m.kv_set_len(0, ctx)), 10)
        us_set = _time_calls(torch, lambda: m.kv_set_len(0, ctx), 20)
        # the same verify writing the hidden states the DFlash draft conditions on
        # (the README's "Architecture": layers 1, 9, 17, 25, 33)
        m.set_taps(DFLASH_TAP_LAYERS)
        us_taps = _time_calls(torch, lambda: (sv.spec_verify_step(m.h, blk, am, ac), m.kv_set_len(0, ctx)), 10)
        m.set_taps([])
        _emit({"suite": "dflash_taps", "config": "qwen3-8b", "ctx": ctx, "n": 16, "layers": DFLASH_TAP_LAYERS,
               "verify_us": round(us_v - us_set, 1), "verify_us_with_taps": round(us_taps - us_set, 1),
               "tap_bytes": len(DFLASH_TAP_LAYERS) * 16 * cfg.d_model * 4})
        for mean in (6.0, 9.0):
            alpha = stepmodel.alpha_for_mean_accept(mean, 15)
            ks = synth.geometric_accept_lengths(64, alpha, 15, stream=int(mean))
            # the rollback of the rejected tail is timed on its own
            def rb():
                for k in ks[:8]:
                    sv.spec_kv_rollback(m.h, 0, ctx + int(k) + 1)
                    m.kv_set_len(0, ctx + 16)
            m.kv_set_len(0, ctx + 16)
            us_rb = (_time_calls(torch, rb, 5) - 8 * us_set) / 8
            toks = float(np.mean(ks + 1))
            t = (us_v - us_set) + max(us_rb, 0.0)
            b = stepmodel.pass_bytes(cfg, 16, ctx)
            _emit({"suite": "dflash", "config": "qwen3-8b", "ctx": ctx, "n": 16, "mean_accept": mean,
                   "alpha": round(alpha, 5), "verify_us": round(us_v - us_set, 1), "rollback_us": round(us_rb, 2),
                   "GBps": round(b / (us_v - us_set) / 1e3, 1), "tokens_per_cycle": round(toks, 3),
                   "tok_s": round(toks / t * 1e6, 1)})
        m.close()
        torch.cuda.empty_cache()


def suite_dflash_block(args):
    """A DFlash-shaped cycle on Qwen3-8B shapes at context 2048 (random
    weights, so timing only): the target's verify of a 16-token block with
    hidden-state taps at layers 1, 9, 17, 25, 33; the draft's context append
    of the m new positions (fc 5*4096 -> 4096, then each draft layer's context
    keys/values); the 5-layer block draft over [last token, mask x 15]; both
    rollbacks.  m = accept + 1 for the mean accept lengths 6 and 9."""
    import numpy as np
    import torch
    import synth
    import speculative_decoding_verify_pass_gb300 as sv
    from speculative_decoding_verify_pass_gb300 import stepmodel
    ctx = 2048
    cfg_t = synth.qwen3_8b(max_ctx=ctx + 64)
    cfg_d = synth.scaled(cfg_t, n_layers=5)
    mt, _ = _model_at_context(cfg_t, ctx)
    md, _ = _model_at_context(cfg_d, ctx)
    taps = mt.set_taps(DFLASH_TAP_LAYERS)
    fc = synth.normal_bf16((cfg_t.d_model, len(DFLASH_TAP_LAYERS) * cfg_t.d_model), 41, 1)
    md.set_context_fc(fc)
    blk_t = torch.tensor(synth.prompt(cfg_t, 16).tolist(), dtype=torch.int32, device="cuda")
    blk_d = torch.tensor([int(blk_t[0])] + [cfg_d.vocab - 1] * 15, dtype=torch.int32, device="cuda")
    am = torch.zeros(16, dtype=torch.int32, device="cuda")
    ac = torch.zeros(1, dtype=torch.int32, device="cuda")
    am2 = torch.zeros(16, dtype=torch.int32, device="cuda")
    ac2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    us_set = _time_calls(torch, lambda: mt.kv_set_len(0, ctx), 20)
    us_verify = _time_calls(torch, lambda: (sv.spec_verify_step(mt.h, blk_t, am, ac), mt.kv_set_len(0, ctx)), 10) - us_set
    us_block = _time_calls(torch, lambda: (sv.spec_verify_step(md.h, blk_d, am2, ac2), md.kv_set_len(0, ctx)), 10) - us_set
    for mean in (6.0, 9.0):
        rows = int(round(mean)) + 1
        us_app = _time_calls(torch, lambda: (sv.spec_context_append(md.h, taps, rows), md.kv_set_len(0, ctx)), 10) - us_set

        def cycle():
            sv.spec_verify_step(mt.h, blk_t, am, ac)
            mt.kv_set_len(0, ctx)
            sv.spec_context_append(md.h, taps, rows)
            sv.spec_verify_step(md.h, blk_d, am2, ac2)
            md.kv_set_len(0, ctx)
        us_cycle = _time_calls(torch, cycle, 10) - 2 * us_set
        alpha = stepmodel.alpha_for_mean_accept(mean, 15)
        ks = synth.geometric_accept_lengths(64, alpha, 15, stream=int(mean))
        toks = float(np.mean(ks + 1))
        _emit({"suite": "dflash_block", "target": "qwen3-8b", "draft": "qwen3-8b-shaped, 5 layers", "ctx": ctx,
               "n": 16, "taps": DFLASH_TAP_LAYERS, "mean_accept": mean, "context_rows": rows,
               "verify_us": round(us_verify, 1), "context_append_us": round(us_app, 1),
               "block_draft_us": round(us_block, 1), "cycle_us": round(us_cycle, 1),
               "tokens_per_cycle": round(toks, 3), "tok_s": round(toks / us_cycle * 1e6, 1)})
    md.check_error()
    mt.check_error()
    mt.close()
    md.close()


def suite_batch(args):
    """Batched sequences: one verify pass over the blocks of nseq independent
    Qwen3-4B sequences at context 2048 (each its own synthetic cache), for
    nseq * n = 16 rows and for n = 4 at nseq = 1, 2, 4.  Weights are read once
    per pass for all sequences; each sequence adds its own KV reads."""
    import torch
    import synth
    import speculative_decoding_verify_pass_gb300 as sv
    from speculative_decoding_verify_pass_gb300 import stepmodel
    ctx, reps = 2048, 10
    cfg = synth.qwen3_4b(max_ctx=ctx + 16 * (reps + 4))
    w = synth.make_weights(cfg)
    m = sv.Model(cfg, w)
    m.batch_reserve(16)
    for l in range(cfg.n_layers):
        k = synth.synthetic_kv(cfg, l, ctx, 0)
        v = synth.synthetic_kv(cfg, l, ctx, 1)
        for q in range(16):
            m.batch_kv_load(q, l, k, v)
    kv_row = 2 * cfg.n_kv_heads * cfg.head_dim * 2
    for nseq, n in ((1, 16), (2, 8), (4, 4), (8, 2), (16, 1), (1, 4), (2, 4)):
        for q in range(nseq):
            m.batch_set_len(q, ctx)
        blocks = torch.tensor([synth.prompt(cfg, n, stream=q).tolist() for q in range(nseq)], dtype=torch.int32,
                              device="cuda")
        am = torch.empty((nseq, n), dtype=torch.int32, device="cuda")
        acc = torch.empty(nseq, dtype=torch.int32, device="cuda")
        for _ in range(3):
            sv.spec_verify_batch(m.h, blocks, am, acc)
        for q in range(nseq):
            m.batch_set_len(q, ctx)
        us = _time_calls(torch, lambda: sv.spec_verify_batch(m.h, blocks, am, acc), reps, warm=0)
        b = stepmodel.pass_bytes(cfg, nseq * n, ctx) + (nseq - 1) * cfg.n_layers * kv_row * ctx
        _emit({"suite": "batch", "config": "qwen3-4b", "ctx": ctx, "nseq": nseq, "n": n, "rows": nseq * n,
               "pass_us": round(us, 1), "bytes": b, "GBps": round(b / us / 1e3, 1),
               "frac_measured_peak": round(b / us / 1e3 / measured_peaks()[0], 3),
               "sequences_per_s": round(nseq / us * 1e6, 1), "rows_per_s": round(nseq * n / us * 1e6, 1)})
    m.check_error()
    m.close()


def suite_shared_prefix(args):
    """The default self-speculative cycle (Qwen3-4B, context 2048, gamma 3,
    50% middle skip) with the draft keeping its own cache for every kept
    layer, then with its leading layers on the target's cache (LayerSkip
    summary 4.3.3): cycle time and the draft cache's size."""
    import torch
    import synth
    import speculative_decoding_verify_pass_gb300 as sv
    cfg, w, plan, m, _ = build_model(args, torch)
    gamma, ctx, steps = args.gamma, args.ctx, 20
    prompt = synth.prompt(cfg, ctx)
    shared = 0
    while shared < len(plan) and plan[shared] == shared:
        shared += 1
    pages = (cfg.max_ctx + 127) // 128 * 2
    slot_bytes = 2 * pages * cfg.n_kv_heads * 64 * cfg.head_dim * 2
    for share in (False, True):
        if share:
            m.share_prefix(True)
        load_synthetic_context(m, cfg, plan, ctx)
        buf = torch.zeros(2 + gamma, dtype=torch.int32, device="cuda")
        buf[0] = int(prompt[-2])
        buf[1] = int(prompt[-1])
        m.kv_set_len(sv.SPEC_CACHE_TARGET, ctx)
        m.kv_set_len(sv.SPEC_CACHE_DRAFT, ctx - 1)
        acc_log = torch.zeros(steps + 4, dtype=torch.int32, device="cuda")
        device_cycles(m, torch, gamma, 3, buf, acc_log, 0)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        device_cycles(m, torch, gamma, steps, buf, acc_log, 3)
        e1.record()
        torch.cuda.synchronize()
        own = len(plan) - (shared if share else 0)
        _emit({"suite": "shared_prefix", "config": args.config, "ctx": ctx, "gamma": gamma, "skip_frac": args.skip,
               "shared_prefix": share, "shared_layers": shared, "draft_cache_slots": own,
               "draft_cache_bytes": own * slot_bytes, "cycle_ms": round(e0.elapsed_time(e1) / steps, 4)})
    m.check_error()
    m.close()


def _expert_op_runs(torch, sv, m, toks, ctx, reps):
    """Per run: (seconds, bytes requested) of the expert operation (gate-up
    and down launches) of every MoE layer of one verify pass, each launch
    bracketed by CUDA events, i.e. run alone."""
    n = len(toks)
    blk = torch.tensor(toks, dtype=torch.int32, device="cuda")
    am = torch.zeros(n, dtype=torch.int32, device="cuda")
    ac = torch.zeros(1, dtype=torch.int32, device="cuda")
    sv.spec_profile_enable(m.h, True)
    sv.spec_verify_step(m.h, blk, am, ac)      # warm the direct-launch path
    sv.spec_kv_rollback(m.h, 0, ctx)
    sv.spec_profile_read(m.h, sv.PROF_ALL)
    out = []
    for _ in range(reps):
        sv.spec_verify_step(m.h, blk, am, ac)
        sv.spec_kv_rollback(m.h, 0, ctx)
        g_ms, g_b, _ = sv.spec_profile_read(m.h, sv.EPI_EXPERT_SWIGLU)
        d_ms, d_b, _ = sv.spec_profile_read(m.h, sv.EPI_EXPERT_DOWN)
        sv.spec_profile_read(m.h, sv.PROF_ALL)
        out.append(((g_ms + d_ms) * 1e-3, g_b + d_b))
    sv.spec_profile_enable(m.h, False)
    return out


def suite_moe(args):
    """DeepSeek-V2-Lite-shaped MoE verify at n = 1..8 with forced synthetic
    routing traces, per-slot against deduplicated expert reads, following the
    MoE page's method (abstract): a step's time is the bytes each kernel
    requests over its effective bandwidth plus fixed time; the bandwidths are
    fitted on one layer's expert operation run alone (a two-layer model of
    the same shapes, launches bracketed by events); bytes from the routing
    traces over those bandwidths predict the time deduplication saves (with
    the bound a bandwidth error puts on it), the crossover, and the best
    draft length over 22 acceptance rates, each beside the measured value."""
    import numpy as np
    import torch
    import synth
    import speculative_decoding_verify_pass_gb300 as sv
    from speculative_decoding_verify_pass_gb300 import stepmodel
    ctx = 2048
    cfg = synth.moe_v2lite(max_ctx=ctx + 64)
    L = cfg.n_layers
    moe_layers = list(range(cfg.first_moe_layer, L))
    trace = synth.routing_trace(L, 16, cfg.n_experts, cfg.top_k)       # [layer][token][k]
    per_expert = stepmodel.expert_bytes(cfg)
    S = cfg.n_shared_experts
    ns = list(range(1, 9))
    modes = ((sv.SPEC_MOE_PER_SLOT, "per_slot"), (sv.SPEC_MOE_DEDUP, "dedup"))

    def layer_bytes(l, n, name):   # expert bytes one layer's expert operation requests
        reads = n * cfg.top_k if name == "per_slot" else stepmodel.union_size(trace[l, :n])
        return (reads + S) * per_expert

    # ---- fit: one layer's expert operation, run alone, at every pass size;
    # per mode, time = t0 + bytes / B (least squares over all runs) ----
    one = synth.scaled(cfg, n_layers=cfg.first_moe_layer + 1)
    m1, _ = _model_at_context(one, ctx)
    ftrace = np.zeros((one.n_layers, 16, cfg.top_k), dtype=np.int32)
    ftrace[cfg.first_moe_layer] = trace[cfg.first_moe_layer]
    m1.force_routing(ftrace)
    pts = {name: ([], []) for _, name in modes}
    for n in ns:
        toks = synth.prompt(cfg, n).tolist()
        for mode, name in modes:
            m1.moe_mode(mode)
            runs = _expert_op_runs(torch, sv, m1, toks, ctx, 5)
            for t, b in runs:
                pts[name][0].append(b)
                pts[name][1].append(t)
            _emit({"suite": "moe_fit_run", "config": "moe-v2-lite", "layer": cfg.first_moe_layer, "n": n,
                   "mode": name, "expert_op_us": round(float(np.mean([t for t, _ in runs])) * 1e6, 2),
                   "bytes": int(runs[0][1])})
    fit = {name: stepmodel.fit_time_model(*pts[name]) for _, name in modes}
    _emit({"suite": "moe_fit", "model": "t = t0 + bytes / B over one layer's expert operation run alone, n = 1..8",
           **{name: {"t0_us": round(f[0] * 1e6, 2), "GBps": round(f[1] / 1e9, 1), "rel_err": round(f[2], 4)}
              for name, f in fit.items()}})
    m1.close()
    del m1
    torch.cuda.empty_cache()

    # ---- measure: the full model ----
    plan = sv.layer_skip_plan(L, 0.5)
    m, _ = _model_at_context(cfg, ctx, plan)
    m.force_routing(trace)
    shared_bytes = len(moe_layers) * S * per_expert
    rows = {}
    for n in ns:
        toks = synth.prompt(cfg, n).tolist()
        u_layers = [stepmodel.union_size(trace[l, :n]) for l in moe_layers]
        for mode, name in modes:
            m.moe_mode(mode)
            us = _verify_us(torch, sv, m, toks, ctx)
            runs = _expert_op_runs(torch, sv, m, toks, ctx, 3)
            exp_us = float(np.mean([t for t, _ in runs])) * 1e6
            exp_bytes = runs[0][1]
            rows[(n, name)] = (us, exp_us, exp_bytes)
            _emit({"suite": "moe", "config": "moe-v2-lite", "ctx": ctx, "n": n, "mode": name,
                   "verify_us": round(us, 1), "expert_us": round(exp_us, 1),
                   "expert_bytes_requested": int(exp_bytes), "routed_bytes_requested": int(exp_bytes - shared_bytes),
                   "expert_GBps": round(exp_bytes / exp_us / 1e3, 1),
                   "unique_experts_mean": round(float(np.mean(u_layers)), 2),
                   "unique_experts_expected": round(stepmodel.union_size_expected(n, cfg.n_experts, cfg.top_k), 2)})

    # ---- predictions: trace bytes of every MoE layer through the fitted model ----
    def expert_time(n, name, scale=1.0):   # seconds, every MoE layer of the pass
        t0, bw, _ = fit[name]
        return stepmodel.model_time(t0, bw * scale, [layer_bytes(l, n, name) for l in moe_layers])

    (_, _, e_ps), (_, _, e_dd) = fit["per_slot"], fit["dedup"]
    saving = []
    for n in ns:
        t_ps, t_dd = expert_time(n, "per_slot"), expert_time(n, "dedup")
        bound = t_ps * e_ps / (1.0 - e_ps) + t_dd * e_dd / (1.0 - e_dd)
        meas = (rows[(n, "per_slot")][0] - rows[(n, "dedup")][0]) * 1e-6
        bps = sum(layer_bytes(l, n, "per_slot") for l in moe_layers)
        bdd = sum(layer_bytes(l, n, "dedup") for l in moe_layers)
        saving.append({"n": n, "byte_share_u": round(bdd / bps, 4),
                       "r_fit": round((bdd / t_dd) / (bps / t_ps), 4),
                       "saving_pred_us": round((t_ps - t_dd) * 1e6, 1), "bound_us": round(bound * 1e6, 1),
                       "saving_meas_us": round(meas * 1e6, 1), "inside_bound": abs(meas - (t_ps - t_dd)) <= bound})
    _emit({"suite": "moe_saving", "points": saving,
           "inside": sum(x["inside_bound"] for x in saving)})
    shares = [x["byte_share_u"] for x in saving]
    r_fit = [x["r_fit"] for x in saving]
    r_meas = [(rows[(n, "dedup")][2] / rows[(n, "dedup")][1]) / (rows[(n, "per_slot")][2] / rows[(n, "per_slot")][1])
              for n in ns]
    measured = next((n for n in ns if rows[(n, "dedup")][0] < rows[(n, "per_slot")][0]), None)
    predicted = stepmodel.first_win(ns, shares, r_fit)
    _emit({"suite": "moe_crossover", "byte_share_u": shares, "r_fit_one_layer_alone": r_fit,
           "r_in_pass": [round(x, 3) for x in r_meas], "crossover_measured": measured,
           "crossover_predicted": predicted})

    # ---- best draft length: from measured verify times, and predicted from
    # operation times (a plain one-token step, the fitted expert operation)
    m.moe_mode(sv.SPEC_MOE_DEDUP)
    t_draft = _draft_us(torch, sv, m, ctx) * 1e-6
    tv_meas = {n: min(rows[(n, "per_slot")][0], rows[(n, "dedup")][0]) * 1e-6 for n in ns}
    pv = {name: stepmodel.predicted_verify_times(rows[(1, name)][0] * 1e-6, lambda n, nm=name: expert_time(n, nm), ns)
          for _, name in modes}
    tv_pred = {n: min(pv["per_slot"][n], pv["dedup"][n]) for n in ns}
    alphas = np.linspace(0.0, 1.0, 22)
    gam = list(range(0, 8))
    st_meas = stepmodel.gamma_staircase(alphas, lambda k: tv_meas[k], t_draft, gam)
    st_pred = stepmodel.gamma_staircase(alphas, lambda k: tv_pred[k], t_draft, gam)
    # how a bandwidth error moves the staircase: every fitted bandwidth at the
    # low and at the high end of its error
    spread = []
    for sgn in (-1.0, 1.0):
        pvs = {name: stepmodel.predicted_verify_times(
                   rows[(1, name)][0] * 1e-6, lambda n, nm=name, sg=sgn: expert_time(n, nm, 1.0 + sg * fit[nm][2]), ns)
               for _, name in modes}
        spread.append(stepmodel.gamma_staircase(alphas, lambda k: min(pvs["per_slot"][k], pvs["dedup"][k]),
                                                t_draft, gam))
    st_free = stepmodel.gamma_staircase(alphas, lambda k: tv_meas[k], 0.0, gam)
    _emit({"suite": "moe_best_gamma", "draft_us": round(t_draft * 1e6, 1), "alphas": 22,
           "best_gamma_measured": st_meas, "best_gamma_predicted": st_pred,
           "best_gamma_predicted_bw_low": spread[0], "best_gamma_predicted_bw_high": spread[1],
           "within_one": sum(abs(a - b) <= 1 for a, b in zip(st_meas, st_pred)),
           "best_gamma_measured_free_draft": st_free,
           "monotone_measured": all(b >= a for a, b in zip(st_meas, st_meas[1:])),
           "monotone_predicted": all(b >= a for a, b in zip(st_pred, st_pred[1:])),
           "verify_us_measured": {n: round(tv_meas[n] * 1e6, 1) for n in ns},
           "verify_us_predicted": {n: round(tv_pred[n] * 1e6, 1) for n in ns}})
    m.close()


def suite_selfspec(args):
    """The MLX self-speculation post's grid on the Qwen3-4B shape at context
    2048 (seeded synthetic KV): for every middle-skip fraction 10..50% and
    draft length 2, 3, 5, device-resident self-speculative cycles against
    plain greedy decoding (one verify of one token per token), timed back to
    back; reports the measured acceptance on the random-init model, the
    verify pass at n = gamma+1 and the draft step."""
    import torch
    import synth
    import speculative_decoding_verify_pass_gb300 as sv
    ctx = args.ctx
    cfg = synth.qwen3_4b(max_ctx=ctx + 1024)
    w = synth.make_weights(cfg)
    m = sv.Model(cfg, w, draft_plan=sv.layer_skip_plan(cfg.n_layers, 0.5))
    kv = [(synth.synthetic_kv(cfg, l, ctx, 0), synth.synthetic_kv(cfg, l, ctx, 1)) for l in range(cfg.n_layers)]
    for l in range(cfg.n_layers):
        m.kv_load(0, l, *kv[l])
    prompt = synth.prompt(cfg, ctx)
    steps = max(args.steps, 8)

    def timed(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3   # s

    # plain greedy: verify n=1 per token; the verify's catch-up pair carries the next input
    pbuf = torch.tensor([int(prompt[-2]), int(prompt[-1])], dtype=torch.int32, device="cuda")
    am1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    ac1 = torch.zeros(1, dtype=torch.int32, device="cuda")

    def plain(k):
        for _ in range(k):
            sv.spec_verify_step(m.h, pbuf[1:2], am1, ac1, None, None, pbuf[0:2])
            sv.spec_kv_rollback(m.h, sv.SPEC_CACHE_TARGET, -1)

    def plain_rate():
        m.kv_set_len(sv.SPEC_CACHE_TARGET, ctx)
        plain(3)
        s = timed(lambda: plain(steps))
        m.check_error()
        return steps / s

    for f in (0.1, 0.2, 0.3, 0.4, 0.5):
        plan = sv.layer_skip_plan(cfg.n_layers, f)
        m.set_draft_plan(plan)
        for i, l in enumerate(plan):
            m.kv_load(1, i, *kv[l])
        m.kv_set_len(sv.SPEC_CACHE_DRAFT, ctx)
        t_draft = _draft_us(torch, sv, m, ctx)
        for gamma in (2, 3, 5):
            n = gamma + 1
            m.kv_set_len(sv.SPEC_CACHE_TARGET, ctx)
            t_verify = _verify_us(torch, sv, m, prompt[:n].tolist(), ctx)
            buf = torch.zeros(2 + gamma, dtype=torch.int32, device="cuda")
            buf[0] = int(prompt[-2])
            buf[1] = int(prompt[-1])
            m.kv_set_len(sv.SPEC_CACHE_TARGET, ctx)
            m.kv_set_len(sv.SPEC_CACHE_DRAFT, ctx - 1)
            acc_log = torch.zeros(steps + 3, dtype=torch.int32, device="cuda")
            device_cycles(m, torch, gamma, 3, buf, acc_log, 0)
            s = timed(lambda: device_cycles(m, torch, gamma, steps, buf, acc_log, 3))
            m.check_error()
            acc = acc_log[3:].cpu().numpy()
            tokens = float(np.sum(acc + 1))
            spec = tokens / s
            base = plain_rate()
            _emit({"suite": "selfspec", "config": cfg.name, "ctx": ctx, "skip_frac": f, "draft_layers": len(plan),
                   "gamma": gamma, "cycles": steps, "accept_mean": round(float(np.mean(acc)), 3),
                   "accept_rate": round(float(np.mean(acc)) / gamma, 4), "tokens_per_cycle": round(tokens / steps, 3),
                   "selfspec_tok_s": round(spec, 1), "plain_tok_s": round(base, 1),
                   "speedup": round(spec / base, 3), "verify_us": round(t_verify, 1), "draft_us": round(t_draft, 1)})
    m.close()


def suite_moe_bytes(args):
    """Expert bytes of one MoE verify pass (n = 8, forced synthetic routing)
    in both modes, for a counter capture: the DeepSeek-V2-Lite shape cut to
    its dense layer 0 and two MoE layers and a 16384-token vocabulary (the
    expert shapes are the full model's; a small device footprint keeps the
    counters' memory save and restore short), context 2048.  Prints per mode the
    analytic bytes each expert launch requests (per slot: one expert read per
    token and slot; dedup: one per distinct expert) and the launch order, so
    that DRAM and L2 counters of the same launches can be set beside them.
    The shared experts are items of the same launches and are counted in
    both the reads and the unique experts.
    Each mode's pass runs inside an NVTX range "timed"."""
    import torch
    import synth
    import speculative_decoding_verify_pass_gb300 as sv
    from speculative_decoding_verify_pass_gb300 import stepmodel
    ctx, n = 2048, 8
    cfg = synth.scaled(synth.moe_v2lite(max_ctx=ctx + 64), n_layers=3, vocab=16384)
    m, _ = _model_at_context(cfg, ctx)
    trace = synth.routing_trace(cfg.n_layers, 16, cfg.n_experts, cfg.top_k)
    m.force_routing(trace)
    toks = synth.prompt(cfg, n).tolist()
    blk = torch.tensor(toks, dtype=torch.int32, device="cuda")
    am = torch.zeros(n, dtype=torch.int32, device="cuda")
    ac = torch.zeros(1, dtype=torch.int32, device="cuda")
    gate_up = 2 * cfg.expert_ffn * cfg.d_model * 2
    down = cfg.expert_ffn * cfg.d_model * 2
    for mode, name in ((sv.SPEC_MOE_PER_SLOT, "per_slot"), (sv.SPEC_MOE_DEDUP, "dedup")):
        m.moe_mode(mode)
        for _ in range(3):
            sv.spec_verify_step(m.h, blk, am, ac)
            sv.spec_kv_rollback(m.h, 0, ctx)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("timed")
        sv.spec_verify_step(m.h, blk, am, ac)
        torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        launches = m.launches()
        sv.spec_kv_rollback(m.h, 0, ctx)
        m.check_error()
        layers = []
        for l in range(cfg.first_moe_layer, cfg.n_layers):
            u = stepmodel.union_size(trace[l, :n])
            reads = (n * cfg.top_k if name == "per_slot" else u) + cfg.n_shared_experts   # + shared, once each
            u += cfg.n_shared_experts
            layers.append({"layer": l, "unique_experts": u, "expert_reads": reads,
                           "gate_up_bytes": reads * gate_up, "down_bytes": reads * down,
                           "unique_gate_up_bytes": u * gate_up, "unique_down_bytes": u * down})
        _emit({"suite": "moe_bytes", "config": cfg.name + ", first 3 layers, vocab 16384", "ctx": ctx, "n": n, "mode": name,
               "launches": launches, "layers": layers})
    m.close()


TRACE_KIND_NAMES = {0: "qkv", 1: "resid", 2: "swiglu", 3: "lm_head", 4: "router", 5: "expert_gate_up",
                    6: "expert_down", 7: "store", 16: "attn_partial", 17: "attn_merge", 18: "embed", 19: "accept"}


TRACE_FIELDS = ("ready_to_exit", "work_to_exit", "gap", "ready_spread", "cta_ready_to_work_med",
                "cta_ready_to_work_max", "work_spread")


def trace_breakdown(stamps, kinds):
    """Per launch kind, from the per-CTA global-timer stamps of one traced
    pass ([ctas][launches][entry, inputs ready, main work done, exit]): mean
    microseconds from the launch's inputs being ready (earliest CTA) to its
    last CTA's exit, from its last main-work stamp to that exit, and from
    the previous launch's last exit to this launch's inputs being ready;
    the spread of the CTAs' ready stamps, the median and largest per-CTA time
    from ready to main work done, and the spread of the main-work stamps;
    plus the pass's span from the first entry to the last exit."""
    out, prev_exit = {}, None
    first, last = None, None
    for l, kind in enumerate(kinds):
        s = stamps[:, l, :]
        live = s[s[:, 0] > 0]
        if len(live) == 0:
            continue
        rd = live[live[:, 1] > 0, 1]
        ready = int(rd.min()) if len(rd) else int(live[:, 0].min())
        wk = live[live[:, 2] > 0, 2]
        ex = int(live[:, 3].max())
        name = TRACE_KIND_NAMES.get(int(kind), str(int(kind)))
        if int(kind) == 1 and l > 0:     # a residual GEMM after the attention merge is the O projection
            name = {17: "o_proj", 2: "down"}.get(int(kinds[l - 1]), name)
        e = out.setdefault(name,
                           {"launches": 0, "ready_to_exit": 0.0, "work_to_exit": 0.0, "gap": 0.0, "gaps": 0,
                            "ready_spread": 0.0, "cta_ready_to_work_med": 0.0, "cta_ready_to_work_max": 0.0,
                            "work_spread": 0.0})
        e["launches"] += 1
        e["ready_to_exit"] += (ex - ready) / 1e3
        if len(rd):
            e["ready_spread"] += (int(rd.max()) - ready) / 1e3
        if len(wk):
            e["work_to_exit"] += (ex - int(wk.max())) / 1e3
            e["work_spread"] += (int(wk.max()) - int(wk.min())) / 1e3
            both = live[(live[:, 1] > 0) & (live[:, 2] > 0)]
            if len(both):
                w = (both[:, 2] - both[:, 1]) / 1e3
                e["cta_ready_to_work_med"] += float(np.median(w))
                e["cta_ready_to_work_max"] += float(w.max())
        if prev_exit is not None:
            e["gap"] += (ready - prev_exit) / 1e3
            e["gaps"] += 1
        prev_exit = ex
        first = int(live[:, 0].min()) if first is None else min(first, int(live[:, 0].min()))
        last = ex if last is None else max(last, ex)
    for e in out.values():
        k = e["launches"]
        for f in ("ready_to_exit", "work_to_exit", "ready_spread", "cta_ready_to_work_med", "cta_ready_to_work_max",
                  "work_spread"):
            e[f] = round(e[f] / k, 2)
        e["gap"] = round(e["gap"] / max(e.pop("gaps"), 1), 2)
    return out, (last - first) / 1e3 if first is not None else 0.0


def suite_trace(args):
    """Where a verify pass's time goes: the launch trace (per-CTA global-timer
    stamps, separate launches) of a verify pass (--config, --ctx; default the
    Qwen3-4B shape at context 2048) for n = 1, 4, 8, 16, summarised per
    launch kind."""
    import torch
    import synth
    import speculative_decoding_verify_pass_gb300 as sv
    ctx = args.ctx
    cfg = synth.PRESETS[args.config](max_ctx=ctx + 64)
    m, _ = _model_at_context(cfg, ctx)
    for n in (1, 4, 8, 16):
        toks = synth.prompt(cfg, n).tolist()
        blk = torch.tensor(toks, dtype=torch.int32, device="cuda")
        am = torch.zeros(n, dtype=torch.int32, device="cuda")
        ac = torch.zeros(1, dtype=torch.int32, device="cuda")
        sv.spec_trace_enable(m.h, True)
        spans, acc = [], {}
        for r in range(4):
            sv.spec_verify_step(m.h, blk, am, ac)
            sv.spec_kv_rollback(m.h, 0, ctx)
            torch.cuda.synchronize()
            if r == 0:
                continue   # first traced pass warms the direct-launch path
            per, span = trace_breakdown(sv.spec_trace_read(m.h), sv.spec_trace_kinds(m.h))
            spans.append(span)
            for k, e in per.items():
                a = acc.setdefault(k, {f: 0.0 for f in TRACE_FIELDS})
                a["launches"] = e["launches"]
                for f in TRACE_FIELDS:
                    a[f] += e[f] / 3
        sv.spec_trace_enable(m.h, False)
        m.check_error()
        for a in acc.values():
            for f in TRACE_FIELDS:
                a[f] = round(a[f], 2)
        _emit({"suite": "trace", "config": cfg.name, "ctx": ctx, "n": n, "traced_pass_us": round(float(np.mean(spans)), 1),
               "verify_us_graph": round(_verify_us(torch, sv, m, toks, ctx), 1), "per_kind_us": acc})
    m.close()


def suite_extras(args):
    """The tiny config (correctness-size model: greedy vs self-speculative
    tokens/s at gamma 4 over the middle-two-of-four plan, verify time per
    pass), the Qwen3-4B prefill of a 2048-token prompt, and plain greedy
    decoding against the self-speculative cycle on the Qwen3-4B shape."""
    import numpy as np
    import torch
    import synth
    import speculative_decoding_verify_pass_gb300 as sv
    # tiny: 128-token prompt, 64 tokens, skip layers {1, 2}, gamma 4
    cfg = synth.tiny()
    w = synth.make_weights(cfg)
    m = sv.Model(cfg, w, draft_plan=[0, 3])
    prompt = synth.prompt(cfg, 128).tolist()
    def reset():
        m.kv_set_len(0, 0)
        m.kv_set_len(1, 0)
    for fn, name in ((lambda: m.greedy(prompt, 64), "greedy"), (lambda: m.selfspec(prompt, 64, 4)[0], "selfspec")):
        reset()
        fn()
        reset()
        torch.cuda.synchronize()
        t0 = time.time()
        out = fn()
        torch.cuda.synchronize()
        dt = time.time() - t0
        _emit({"suite": "extras", "what": "tiny_" + name, "tokens": len(out), "wall_s": round(dt, 4),
               "tok_s_host_loop": round(len(out) / dt, 1)})
    reset()
    m.prefill(prompt)
    us = _verify_us(torch, sv, m, prompt[:5], 128)
    _emit({"suite": "extras", "what": "tiny_verify_n5", "ctx": 128, "us": round(us, 1)})
    m.close()
    # Qwen3-4B: prefill of 2048 tokens; plain greedy decode vs the self-speculative cycle
    cfg = synth.qwen3_4b(max_ctx=2048 + 1024)
    plan = sv.layer_skip_plan(cfg.n_layers, 0.5)
    w = synth.make_weights(cfg)
    m = sv.Model(cfg, w, draft_plan=plan)
    prompt = synth.prompt(cfg, 2048).tolist()
    m.prefill(prompt)
    torch.cuda.synchronize()
    for _ in range(2):
        m.kv_set_len(0, 0)
        m.kv_set_len(1, 0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        m.prefill(prompt)
        e1.record()
        torch.cuda.synchronize()
    _emit({"suite": "extras", "what": "qwen3-4b_prefill", "tokens": 2048, "ms": round(e0.elapsed_time(e1), 2),
           "tok_s": round(2048 / (e0.elapsed_time(e1) / 1e3), 1)})
    ctx = m.kv_len(0)
    us1 = _verify_us(torch, sv, m, prompt[:1], ctx)
    _emit({"suite": "extras", "what": "qwen3-4b_plain_greedy", "ctx": ctx, "us_per_token": round(us1, 1),
           "tok_s": round(1e6 / us1, 1)})
    m.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="geometric", choices=["geometric", "selfspec"])
    ap.add_argument("--config", default=None, help="model preset (default llama-3.1-8b; selfspec: qwen3-4b)")
    ap.add_argument("--n", type=int, default=8, help="geometric: verify block size (last accepted + n-1 drafts)")
    ap.add_argument("--alpha", type=float, default=0.7, help="geometric: probability that a draft is clean")
    ap.add_argument("--gamma", type=int, default=3, help="selfspec: draft steps per cycle")
    ap.add_argument("--skip", type=float, default=0.5, help="selfspec: middle-skip fraction of the draft")
    ap.add_argument("--ctx", type=int, default=None, help="KV context (default 4096; selfspec: 2048)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="keep only the first N layers (a smaller case for counter captures; the line names it)")
    ap.add_argument("--suite", default=None, choices=["sweep", "geometric", "dflash", "dflash_block", "batch", "shared_prefix", "moe", "moe_bytes",
                             "selfspec", "trace", "extras"],
                    help="run one measurement suite instead of the default bench line")
    args = ap.parse_args()
    if args.config is None:
        args.config = "qwen3-4b" if args.workload == "selfspec" or args.suite else "llama-3.1-8b"
    if args.ctx is None:
        args.ctx = 2048 if args.workload == "selfspec" or args.suite else 4096
    if args.suite:
        import __graft_entry__
        __graft_entry__.build()
        {"sweep": suite_sweep, "geometric": suite_geometric, "dflash": suite_dflash,
         "dflash_block": suite_dflash_block, "batch": suite_batch, "shared_prefix": suite_shared_prefix,
         "moe": suite_moe, "moe_bytes": suite_moe_bytes, "selfspec": suite_selfspec,
         "trace": suite_trace,
         "extras": suite_extras}[args.suite](args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
