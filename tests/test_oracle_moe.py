"""Pins of the oracle's MoE layer, router and stack.

The layer follows the "llm-decoding" post (§"The exact architecture": top-8 of
128 routed experts plus one always-on shared expert, hidden 2816, FFN 704;
§"Where the 7.36 GB goes": gate/up/down 2816x704 per expert) with the softmax
top-k router, GELU-tanh gating and per-row E4M3 weights that the benchmark
configurations fix. Each pin compares the oracle with a computation that does
not share its formulation: a dense evaluation of every expert with a masked
weight vector (torch fp64, torch's own E4M3 decode), a plain GeGLU MLP, exact
identities, and batch invariance.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import bf16_values, dequant_torch, to_oracle_layer

SMALL = dict(hidden=64, ffn=16, experts=16)


def _small_layer(seed, s=0.0, k=4, zero_shared=False):
    p = synth.layer(seed, s=s, zero_shared=zero_shared, **SMALL)
    return p, to_oracle_layer(p, k=k)


def _dense_reference(p, L, x, k):
    """Every expert evaluated densely in torch fp64, then combined with a weight
    vector that is the renormalised softmax over the top-k logits and 0 elsewhere."""
    E = L.router_w.shape[0]
    wr = p["router_w"].to(torch.float64)
    xt = torch.from_numpy(x)
    logits = xt @ wr.T
    if p["router_b"] is not None:
        logits = logits + p["router_b"].to(torch.float64)
    top = torch.topk(logits, k, dim=1)
    sel = torch.softmax(top.values, dim=1)       # renormalised top-k == softmax of the top-k logits
    mask = torch.zeros_like(logits).scatter_(1, top.indices, sel)
    g = torch.einsum("efh,mh->mef", dequant_torch(L.gate_q, L.gate_s), xt)
    u = torch.einsum("efh,mh->mef", dequant_torch(L.up_q, L.up_s), xt)
    a = torch.nn.functional.gelu(g, approximate="tanh") * u
    d = torch.einsum("ehf,mef->meh", dequant_torch(L.down_q, L.down_s), a)
    y = (mask.unsqueeze(-1) * d[:, :E]).sum(1) + d[:, E:].sum(1)
    return y.numpy(), top.indices.numpy(), sel.numpy(), logits.numpy()


@pytest.mark.parametrize("seed,s,k,M", [(11, 0.0, 4, 3), (12, 1.1, 4, 5), (13, 2.0, 2, 8), (14, 0.0, 16, 2)])
def test_layer_matches_dense_masked_evaluation(seed, s, k, M):
    p, L = _small_layer(seed, s=s, k=k)
    x = bf16_values(synth.hidden_states(seed + 100, M, hidden=SMALL["hidden"]))
    out = oracle.moe_layer(L, x)
    y_ref, ids_ref, w_ref, logits_ref = _dense_reference(p, L, x, k)
    np.testing.assert_allclose(out.y, y_ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_array_equal(out.ids, ids_ref)
    np.testing.assert_allclose(out.w, w_ref, rtol=1e-12)
    np.testing.assert_allclose(out.logits, logits_ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(out.w.sum(axis=1), 1.0, rtol=1e-14)
    srt = np.sort(logits_ref, axis=1)[:, ::-1]
    if k < L.router_w.shape[0]:
        np.testing.assert_allclose(out.margin, srt[:, k - 1] - srt[:, k], rtol=1e-9, atol=1e-14)


def test_single_expert_is_a_plain_geglu_mlp():
    """E = 1, k = 1 and a zero shared expert: the layer is down(gelu(gate x) * up x)."""
    p = synth.layer(21, hidden=48, ffn=24, experts=1, zero_shared=True)
    L = to_oracle_layer(p, k=1)
    x = bf16_values(synth.hidden_states(22, 4, hidden=48))
    out = oracle.moe_layer(L, x)
    xt = torch.from_numpy(x)
    wg = dequant_torch(L.gate_q[0], L.gate_s[0])
    wu = dequant_torch(L.up_q[0], L.up_s[0])
    wd = dequant_torch(L.down_q[0], L.down_s[0])
    mlp = torch.nn.functional.linear(
        torch.nn.functional.gelu(xt @ wg.T, approximate="tanh") * (xt @ wu.T), wd)
    np.testing.assert_allclose(out.y, mlp.numpy(), rtol=1e-12, atol=1e-14)
    assert (out.ids == 0).all() and (out.w == 1.0).all()


def test_shared_expert_enters_with_weight_one():
    p, L = _small_layer(31)
    x = bf16_values(synth.hidden_states(32, 2, hidden=SMALL["hidden"]))
    out = oracle.moe_layer(L, x)
    for t in range(2):
        routed = sum(out.w[t, i] * oracle.expert_token(L, out.ids[t, i], x[t]) for i in range(L.k))
        shared = oracle.expert_token(L, SMALL["experts"], x[t])
        np.testing.assert_allclose(out.y[t], routed + shared, rtol=1e-12, atol=1e-15)


def test_router_one_hot_input_reads_one_column():
    """x = e_j makes every logit the bf16 weight W_r[e, j] (plus bias): a transposed
    or mis-strided router would read another element."""
    p, L = _small_layer(41, s=1.1)
    H = SMALL["hidden"]
    for j in (0, 5, H - 1):
        x = np.zeros(H)
        x[j] = 1.0
        ids, w, margin, logits = oracle.router_token(L, x)
        expect = bf16_values(p["router_w"])[:, j] + p["router_b"].double().numpy()
        np.testing.assert_array_equal(logits, expect)


def test_router_ties_go_to_lower_index():
    H, E = 8, 6
    wr = torch.zeros((E, H), dtype=torch.bfloat16)
    wr[:, 0] = torch.tensor([1.0, 2.0, 2.0, 0.5, 2.0, 1.0])
    p = synth.layer(1, hidden=H, ffn=4, experts=E)
    p["router_w"] = wr
    L = to_oracle_layer(p, k=2)
    x = np.zeros(H)
    x[0] = 1.0
    ids, w, margin, _ = oracle.router_token(L, x)
    assert list(ids) == [1, 2] and margin == 0.0
    np.testing.assert_allclose(w, [0.5, 0.5], rtol=1e-15)


def test_batch_invariance():
    """Tokens never interact inside a layer: row i of an M-token call equals the
    call on token i alone."""
    p, L = _small_layer(51, s=1.1)
    x = bf16_values(synth.hidden_states(52, 6, hidden=SMALL["hidden"]))
    full = oracle.moe_layer(L, x)
    for i in range(6):
        one = oracle.moe_layer(L, x[i:i + 1])
        np.testing.assert_array_equal(one.y[0], full.y[i])
        np.testing.assert_array_equal(one.ids[0], full.ids[i])


def test_stack_layer_is_residual_of_normed_layer():
    p, L = _small_layer(61, s=1.1)
    h = bf16_values(synth.hidden_states(62, 3, hidden=SMALL["hidden"])) * 3.0
    out = oracle.stack_layer(L, h, eps=1e-6)
    rms = np.sqrt((h ** 2).mean(axis=1, keepdims=True) + 1e-6)
    ref = oracle.moe_layer(L, h / rms)
    np.testing.assert_allclose(out.y, h + ref.y, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(out.ids, ref.ids)
    # iterating stays batch invariant
    h2 = out.y
    for _ in range(3):
        h2 = oracle.stack_layer(L, h2).y
    h1 = h[1:2]
    for _ in range(4):
        h1 = oracle.stack_layer(L, h1).y
    np.testing.assert_array_equal(h1[0], h2[1])


def test_zipf_bias_gives_the_expected_sharing():
    """With the full-size router (128 x 2816, N(0, 0.02)) and 5 N(0,1) tokens, the
    bias -s ln(e+1) must give the sharing the benchmark configuration expects:
    about 35 unique experts without bias and 15-26 at s = 1.1."""
    g = torch.Generator().manual_seed(7)
    wr = (torch.randn((128, 2816), generator=g) * 0.02).to(torch.bfloat16)
    uniq = {0.0: [], 1.1: [], 2.0: []}
    for s in uniq:
        b = synth.zipf_bias(s) if s else None
        p = {"router_w": wr, "router_b": b}
        L = oracle.LayerParams(
            router_w=wr.view(torch.int16).numpy().view(np.uint16),
            router_b=None if b is None else b.numpy(),
            gate_q=np.zeros((129, 1, 2816), np.uint8), gate_s=np.ones((129, 1), np.float32),
            up_q=np.zeros((129, 1, 2816), np.uint8), up_s=np.ones((129, 1), np.float32),
            down_q=np.zeros((129, 2816, 1), np.uint8), down_s=np.ones((129, 2816), np.float32))
        for trial in range(12):
            x = bf16_values(synth.hidden_states(1000 + trial, 5))
            ids = np.stack([oracle.router_token(L, x[t])[0] for t in range(5)])
            uniq[s].append(len(np.unique(ids)))
    assert 30 <= np.mean(uniq[0.0]) <= 40
    assert 15 <= np.mean(uniq[1.1]) <= 26
    assert np.mean(uniq[2.0]) < np.mean(uniq[1.1]) < np.mean(uniq[0.0])
