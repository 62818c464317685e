"""Benchmark of the speculative-decoding verify pass on one GB300 (or N replicas).

One step = one greedy self-speculative cycle of the Qwen3-4B-shaped target
(random-init bf16 weights, prompt of 2048 random ids): gamma draft steps over
the middle-skip layer plan (the first with the catch-up pair, n=2), one
verify pass of n = gamma+1 tokens over all 36 layers with argmax and the
cumulative-product accept, and the device-side rollback of both caches.
The loop stays on the device (token ids never visit the host).

Printed JSON line: accepted tokens/s (the MLX post's and the DFlash README's
throughput metric), the verify pass's time and HBM bandwidth against 8 TB/s,
a roofline entry for the streaming GEMM (the dominant kernel), an end-to-end
figure through the host-driven API with pinned host copies, the oracle's
rate on the host cores, and the SM clocks seen during the timed region.

    python bench.py [--steps K] [--warmup W] [--gamma 3] [--skip 0.5]
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


def pass_bytes(cfg, n, ctx, plan=None):
    """Algorithmic bytes of one dense pass: executed layers' weights, LM head,
    KV read over ctx, KV rows written, embedding rows."""
    plan = list(range(cfg.n_layers)) if plan is None else plan
    d, hd = cfg.d_model, cfg.head_dim
    qw, kw = cfg.n_heads * hd, cfg.n_kv_heads * hd
    per_layer = ((qw + 2 * kw) * d + d * qw + 3 * cfg.ffn_dim * d) * 2
    kv = 2 * kw * 2
    return len(plan) * (per_layer + kv * (ctx + n)) + cfg.vocab * d * 2 + n * d * 2


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def build_model(args, torch):
    import synth
    import speculative_decoding_verify_pass_gb300 as sv
    cfg = synth.PRESETS[args.config](max_ctx=args.ctx + 1024)
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


def run_native(args):
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
    e0.record(stream)
    launches = device_cycles(m, torch, gamma, args.steps, buf, acc_log, args.warmup)
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = clk.stop()
    ms = e0.elapsed_time(e1)
    m.check_error()
    accepts = acc_log[args.warmup:total].cpu().numpy()
    tokens = float(np.sum(accepts + 1))
    if dist:
        t = torch.tensor([ms, tokens], dtype=torch.float64, device="cuda")
        mx = t.clone()
        dist.all_reduce(mx, op=dist.ReduceOp.MAX)
        sm_ = t.clone()
        dist.all_reduce(sm_, op=dist.ReduceOp.SUM)
        ms, tokens = float(mx[0]), float(sm_[1])
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
    gms, gbytes, glaunch = sv.spec_profile_read(m.h)
    sv.spec_profile_enable(m.h, False)
    peak, peak_kind = measured_peaks()
    achieved = gbytes / (gms / 1e3) / 1e9 if gms > 0 else 0.0

    # ---- end to end through the host-driven API (pinned copies each step) ----
    e2e = run_e2e(m, torch, sv, gamma, args, prompt, ctx_now)

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "%s self-speculative cycle at context %d (seeded synthetic KV): %d draft steps over the "
                               "%d%% middle-skip plan (%d of %d layers) + verify n=%d + accept + rollback" % (
                                   cfg.name, ctx, gamma, round(args.skip * 100), len(plan), cfg.n_layers, n),
                   "model": cfg.name + "-shaped, random-init N(0,0.02) bf16", "global_batch": world, "seq_len": ctx,
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
                     "frac": round(achieved / peak, 4), "traffic": None,
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


def cpu_baseline(cfg, w, plan, args, prompt):
    import oracle
    orc, tc, dc = oracle_cycle_setup(cfg, w, plan, args.ctx)
    t0 = time.perf_counter()
    toks = oracle_cycle(orc, tc, dc, plan, args.gamma, args.ctx, int(prompt[-1]))
    dt = time.perf_counter() - t0
    return {"value": round(toks / dt, 4), "unit": "tok/s", "cores": oracle.get_threads(), "kind": "oracle",
            "sample": "one cycle (%d draft passes + verify n=%d) at context %d on synthetic seeded KV, "
                      "fp32 C oracle, %.1f s" % (args.gamma, args.gamma + 1, args.ctx, dt)}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    import synth
    import speculative_decoding_verify_pass_gb300 as sv  # layer plan rule only
    oracle.build()
    synth.build()
    cfg = synth.PRESETS[args.config](max_ctx=args.ctx + 64)
    w = synth.make_weights(cfg)
    plan = sv.layer_skip_plan(cfg.n_layers, args.skip)
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--config", default="qwen3-4b")
    ap.add_argument("--gamma", type=int, default=3)
    ap.add_argument("--skip", type=float, default=0.5)
    ap.add_argument("--ctx", type=int, default=2048)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
