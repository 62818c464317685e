"""Shared fixtures.  `-m gpu` tests need a CUDA device; the rest run on CPU."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def tiny_cfg():
    import synth
    return synth.tiny()


@pytest.fixture(scope="session")
def tiny_weights(tiny_cfg):
    import synth
    return synth.make_weights(tiny_cfg)


@pytest.fixture(scope="session")
def tiny_oracle(tiny_cfg, tiny_weights):
    import oracle
    return oracle.Oracle(tiny_cfg, tiny_weights)


@pytest.fixture(scope="session")
def tiny_prompt(tiny_cfg):
    import synth
    return synth.prompt(tiny_cfg, 128)


def small_moe_cfg():
    """A MoE model small enough for pure-oracle checks (shape family of the
    DeepSeek-V2-Lite-like preset: dense layer 0, routed + shared experts)."""
    import synth
    return synth.ModelConfig("moe-small", 3, 128, 2, 2, 64, 256, 512, rope_theta=1e4,
                             n_experts=8, top_k=2, expert_ffn=64, n_shared_experts=2,
                             first_moe_layer=1, max_ctx=256, index=4)


def small_gqa_cfg():
    """A small grouped-query model (4 query heads per kv head, tied LM head)."""
    import synth
    return synth.ModelConfig("gqa-small", 3, 256, 8, 2, 64, 512, 1000, rope_theta=5e5,
                             tied_embeddings=True, max_ctx=512, index=1)
