"""The byte accounting used for the roofline reproduces the byte budget that the
"llm-decoding" post hand-counts from the config shapes (§"Where the 7.36 GB
goes"), and gives the FP8 step sizes used as the roofline numerator."""

import os

import pytest

from fine_grained_moe_gb300 import traffic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "byte_budget.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_page_byte_budget_in_bf16():
    g = _golden()
    layers = 30
    experts = layers * 8 * traffic.expert_bytes(weight_bytes=2, with_scales=False)
    assert experts / 1e9 == pytest.approx(g["experts_gb"], abs=0.01)
    assert experts / 2 / 1e9 == pytest.approx(g["experts_params_b"], abs=0.005)
    assert traffic.lm_head_bytes() / 1e9 == pytest.approx(g["lm_head_gb"], abs=0.005)
    assert traffic.lm_head_bytes() / 2 / 1e6 == pytest.approx(g["lm_head_params_m"], abs=0.5)
    router = layers * traffic.router_bytes(with_bias=False)
    assert router / 1e9 == pytest.approx(g["router_gb"], abs=0.005)
    dense = layers * 3 * 2816 * 2112
    assert dense / 1e6 == pytest.approx(g["dense_mlp_params_m"], abs=0.5)
    assert dense * 2 / 1e9 == pytest.approx(g["dense_mlp_gb"], abs=0.005)
    total = experts + router + traffic.lm_head_bytes() + dense * 2 + g["attention_gb"] * 1e9
    assert total / 1e9 == pytest.approx(g["total_gb"], abs=0.02)
    floor_ms = g["total_gb"] / g["a100_hbm_tbs"]
    assert floor_ms == pytest.approx(g["floor_ms"], abs=0.05)
    assert 1000.0 / floor_ms == pytest.approx(g["ceiling_tok_s"], abs=2)


def test_fp8_step_sizes():
    # M = 1: 8 routed experts per layer
    b1 = traffic.step_bytes([8] * 30)
    assert b1 == 30 * (9 * 5964288 + 721408) + 1476395008
    assert b1 / 1e9 == pytest.approx(3.11, abs=0.01)   # 30 x 54.4 MB + 1.476 GB
    assert traffic.step_bytes([20] * 30) / 1e9 == pytest.approx(5.26, abs=0.01)
    assert traffic.step_bytes([35] * 30) / 1e9 == pytest.approx(7.94, abs=0.01)
    # one C0-size layer, no lm_head
    assert traffic.step_bytes([8], with_lm_head=False, with_bias=False) == 9 * 5964288 + 720896


def test_fp8_lm_head_halves_the_embedding_bytes():
    # 262,144 x 2816 codes + one fp32 scale per row; the page's 738M-parameter
    # projection at one byte each (§"Where the 7.36 GB goes")
    g = _golden()
    b = traffic.lm_head_fp8_bytes()
    assert b == 262144 * 2816 + 4 * 262144
    assert (b - 4 * 262144) / 1e6 == pytest.approx(g["lm_head_params_m"], abs=0.5)
    assert traffic.lm_head_bytes() - b == 262144 * (2816 - 4)
    assert (traffic.step_bytes([20] * 30, fp8_lm_head=True)
            == traffic.step_bytes([20] * 30) - traffic.lm_head_bytes() + b)


def test_dense_step_replaces_the_shared_expert_by_the_mlp():
    # per layer: the distinct routed experts, the 2816 x 2112 MLP (E4M3 + fp32
    # row scales 2 x 2112 + 2816) and the router; no shared expert
    mlp = 3 * 2816 * 2112 + 4 * (2 * 2112 + 2816)
    assert traffic.dense_mlp_bytes() == mlp
    assert (traffic.step_bytes([20] * 30, dense_width=2112)
            == 30 * (20 * 5964288 + mlp + 721408) + 1476395008)
    assert (traffic.step_bytes([20] * 30, dense_width=2112) - traffic.step_bytes([20] * 30)
            == 30 * (mlp - 5964288))
