"""Writes tiny_greedy.txt: plain greedy tokens of the tiny decoder, computed
by the CPU oracle only (synth inputs: weights seed 1234, prompt seed 1,
128 prompt tokens, 64 generated tokens).

    python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth   # noqa: E402


def main():
    cfg = synth.tiny()
    orc = oracle.Oracle(cfg, synth.make_weights(cfg))
    toks = oracle.greedy_generate(orc, synth.prompt(cfg, 128), 64)
    with open(os.path.join(HERE, "tiny_greedy.txt"), "w") as f:
        f.write("# plain greedy continuation of the tiny decoder (oracle), 64 tokens\n")
        f.write(" ".join(str(t) for t in toks) + "\n")


if __name__ == "__main__":
    main()
