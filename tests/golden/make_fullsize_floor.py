"""Writes fullsize_floor.txt: how far the fp32-accumulating oracle drifts from
the fp64-accumulating build of the same definition, per full-size workload.

Both builds share every bf16 rounding point; they differ only in the
precision of the long sums.  Small differences in those sums flip bf16
roundings, the flips feed the residual stream of later layers, and the logit
rows drift apart with depth.  The stored statistics are the reproducibility
floor of fp32 accumulation for each workload; the full-size GPU tests bound
the GPU's deviation from the fp64 build by them.

Each case: the preset model at full size, synthetic KV for `ctx` positions in
every layer (synth.synthetic_kv), then one verify pass of `n` prompt tokens
(synth.prompt, given stream).  `layers` < the preset's depth truncates the
model to its first layers (a full-width shallow case).  MoE cases force both
builds onto the fp64 build's own routing so that routing does not enter the
logit comparison; for them two more figures are stored: the share of
(MoE layer, token, slot) choices on which the two builds' free routings
differ, and the largest router-probability difference between the builds
under that forced routing.  Computed by the CPU oracle only.

    python tests/golden/make_fullsize_floor.py [case ...]

With case names, only those cases are computed and their lines replaced or
appended; the other lines of the file are kept.
"""
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth   # noqa: E402

# name, preset, layers (0: all), ctx, n, prompt stream
CASES = [
    ("qwen3-4b-L1", "qwen3-4b", 1, 128, 16, 7),
    ("llama-3.1-8b-L1", "llama-3.1-8b", 1, 128, 16, 7),
    ("qwen3-4b", "qwen3-4b", 0, 2048, 4, 7),
    ("qwen3-4b-n6", "qwen3-4b", 0, 2048, 6, 11),
    ("llama-3.1-8b", "llama-3.1-8b", 0, 4096, 8, 7),
    ("qwen3-8b", "qwen3-8b", 0, 2048, 16, 7),
    ("moe-v2-lite", "moe-v2-lite", 0, 2048, 4, 9),
    ("llama-3.1-8b-n1", "llama-3.1-8b", 0, 4096, 1, 13),
    ("moe-v2-lite-n8", "moe-v2-lite", 0, 2048, 8, 15),
]

ATOL = RTOL = 2e-2


def case_config(preset, layers, ctx, n):
    cfg = synth.PRESETS[preset](max_ctx=ctx + 64)
    if layers:
        cfg = synth.scaled(cfg, n_layers=layers)
    return cfg


def load_context(orc, cache, cfg, ctx):
    for l in range(cfg.n_layers):
        k = synth.synthetic_kv(cfg, l, ctx, 0)
        v = synth.synthetic_kv(cfg, l, ctx, 1)
        cache.load(l, k.reshape(ctx, -1), v.reshape(ctx, -1))
    cache.set_len(ctx)


def floor_stats(a, b):
    """Deviation of logits a from logits b: mean |a-b|, max |a-b|, share of
    entries outside ATOL + RTOL*|b|."""
    e = np.abs(a.astype(np.float64) - b.astype(np.float64))
    return float(e.mean()), float(e.max()), float(np.mean(e > ATOL + RTOL * np.abs(b)))


def run_case(preset, layers, ctx, n, stream):
    """(mean, max, share) of the logits, plus (routing mismatch share, max
    router-probability difference) for MoE models, else None."""
    cfg = case_config(preset, layers, ctx, n)
    w = synth.make_weights(cfg)
    toks = synth.prompt(cfg, n, stream=stream)
    moe = cfg.n_experts > 0
    shape = (cfg.n_layers, n, cfg.n_experts)
    builds = {}
    for acc64 in (True, False):
        orc = oracle.Oracle(cfg, w, acc64=acc64)
        cache = orc.new_cache()
        load_context(orc, cache, cfg, ctx)
        free_ids = forced = probs = None
        if moe:
            _, free_ids, _ = orc.forward(cache, orc.full_plan, toks, ctx, logits_from=None, want_routing=True)
            cache.truncate(ctx)
            forced = np.maximum(builds[True][1], 0) if not acc64 else np.maximum(free_ids, 0)
            probs = np.zeros(shape, np.float32)
        logits, _, _ = orc.forward(cache, orc.full_plan, toks, ctx, want_routing=moe, forced_ids=forced, probs=probs)
        builds[acc64] = (logits, free_ids, probs)
        del orc, cache
    (ref, ids64, p64), (got, ids32, p32) = builds[True], builds[False]
    route = None
    if moe:
        route = (float(np.mean(ids32[cfg.first_moe_layer:] != ids64[cfg.first_moe_layer:])),
                 float(np.max(np.abs(p32.astype(np.float64) - p64))))
    return floor_stats(got, ref), route


def main(only=None):
    out = os.path.join(HERE, "fullsize_floor.txt")
    header = ["# fp32-accumulating oracle vs the fp64-accumulating build, same inputs and rounding points",
              "# written by make_fullsize_floor.py (CPU oracle only); tolerance %g abs + %g rel" % (ATOL, RTOL),
              "# name preset layers ctx n stream mean_abs max_abs share_outside route_mismatch route_max_dp"]
    kept = {}
    if only and os.path.exists(out):
        for line in open(out):
            if line.strip() and line[0] != "#":
                kept[line.split()[0]] = line.rstrip("\n")
    for name, preset, layers, ctx, n, stream in CASES:
        if only and name not in only:
            continue
        t = time.time()
        (mean, mx, share), route = run_case(preset, layers, ctx, n, stream)
        tail = "%.6g %.6g" % route if route else "- -"
        kept[name] = "%s %s %d %d %d %d %.6g %.6g %.6g %s" % (name, preset, layers, ctx, n, stream, mean, mx, share,
                                                              tail)
        print(kept[name], "(%.0f s)" % (time.time() - t), flush=True)
    order = [c[0] for c in CASES if c[0] in kept]
    with open(out, "w") as f:
        f.write("\n".join(header + [kept[k] for k in order]) + "\n")


if __name__ == "__main__":
    main(sys.argv[1:] or None)
