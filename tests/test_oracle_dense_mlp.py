"""Pins of the oracle's always-on dense MLP (the wider shared-MLP variant).

The byte list of "llm-decoding" (§"Where the 7.36 GB goes") counts an
always-on dense MLP of 2816 x 2112 per layer, three times the 704 width of a
routed expert. The oracle computes it as a gated-GELU MLP of width 2112 with
per-row E4M3 weights. Pins: the MLP against a plain GeGLU MLP in torch fp64
(torch's own float8 decode); the closed-form identity that a gated MLP of
width 3F is the sum of three width-F MLPs over its column blocks when the
down rows keep their full-width scales (the layout a kernel can stream as
three shared experts); and a layer with the dense MLP equals its routed part
plus that MLP, with unchanged routing.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import bf16_values, dequant_torch, to_oracle_layer


def _mlp(p):
    return oracle.MlpParams(**{k: p[k].numpy() for k in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")})


def test_dense_mlp_is_a_plain_geglu_mlp():
    H, W = 96, 72
    p = synth.dense_mlp(41, width=W, hidden=H)
    x = bf16_values(synth.hidden_states(42, 1, hidden=H))[0]
    got = oracle.mlp_token(_mlp(p), x)
    xt = torch.from_numpy(x)
    g = dequant_torch(p["gate_q"].numpy(), p["gate_s"].numpy()) @ xt
    u = dequant_torch(p["up_q"].numpy(), p["up_s"].numpy()) @ xt
    a = torch.nn.functional.gelu(g, approximate="tanh") * u
    ref = dequant_torch(p["down_q"].numpy(), p["down_s"].numpy()) @ a
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-11, atol=1e-15)


@pytest.mark.parametrize("W,F", [(72, 24), (2112, 704)])
def test_width_3f_mlp_is_the_sum_of_its_three_column_blocks(W, F):
    H = 96 if W == 72 else 2816
    p = synth.dense_mlp(43, width=W, hidden=H)
    parts = synth.dense_mlp_as_experts(p, ffn=F)
    assert parts["gate_q"].shape == (W // F, F, H) and parts["down_q"].shape == (W // F, H, F)
    x = bf16_values(synth.hidden_states(44, 1, hidden=H))[0]
    whole = oracle.mlp_token(_mlp(p), x)
    split = sum(oracle.mlp_token(_mlp({k: v[i] for k, v in parts.items()}), x) for i in range(W // F))
    np.testing.assert_allclose(split, whole, rtol=1e-11, atol=1e-13 * np.abs(whole).max())


def test_layer_with_dense_shared_is_routed_part_plus_the_mlp():
    H, F, E = 64, 16, 16
    lay = synth.layer(45, hidden=H, ffn=F, experts=E, n_shared=0, s=1.1)
    L = to_oracle_layer(lay, k=4, n_shared=0)
    p = synth.dense_mlp(46, width=3 * F, hidden=H)
    x = bf16_values(synth.hidden_states(47, 3, hidden=H))
    base = oracle.moe_layer(L, x)
    dense = oracle.moe_layer(L, x, dense_shared=_mlp(p))
    np.testing.assert_array_equal(dense.ids, base.ids)
    np.testing.assert_array_equal(dense.margin, base.margin)
    extra = np.stack([oracle.mlp_token(_mlp(p), x[t]) for t in range(3)])
    np.testing.assert_allclose(dense.y, base.y + extra, rtol=1e-12, atol=1e-15)
