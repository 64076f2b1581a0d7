"""Pins of the oracle's speculative sampling verify at temperature T > 0.

"llm-decoding" (§"What we learned") states the property: a drafted token is
kept only if it passes the distribution the full model samples from, a
rejected one falls back to a real model step, and the output distribution is
that of ordinary decoding. With a drafter that proposes tokens only (one-hot
proposals), the oracle accepts d_i when u < p_i(d_i) and otherwise samples p_i
with d_i removed. The pins: a worked example by hand; the T -> 0 limit is the
greedy rule; the emitted token's distribution equals the target's own
distribution (quadrature over the uniforms: the lossless property); the
inverse CDF against numpy's cumulative sum; the logits against torch.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import bf16_bits, bf16_values


def test_worked_example_by_hand():
    # position 0: z = (0, 1, 2), T = 1: p = e^z / (1 + e + e^2) = (0.0900, 0.2447, 0.6652)
    # position 1: z = (1, 0, 0): p = (e, 1, 1) / (e + 2) = (0.5761, 0.2119, 0.2119)
    z = np.array([[0.0, 1.0, 2.0], [1.0, 0.0, 0.0]])
    e = np.e
    p0 = np.array([1.0, e, e * e]) / (1 + e + e * e)
    p1 = np.array([e, 1.0, 1.0]) / (e + 2)
    # draft 2 accepted (0.1 < p0[2]); then p1 sampled at 0.5 -> token 0 (p1[0] > 0.5)
    a, tok, mg, gap = oracle.spec_sample(z, 1.0, [2], [0.1], [0.5, 0.5])
    assert (a, tok) == (1, 0)
    assert mg == pytest.approx(p0[2] - 0.1, rel=1e-12) and gap == pytest.approx(p1[0] - 0.5, rel=1e-12)
    # draft 0 rejected (0.9 >= p0[0]); residual (0, p0[1], p0[2]) renormalised, at 0.5 -> token 2
    a, tok, mg, gap = oracle.spec_sample(z, 1.0, [0], [0.9], [0.5, 0.5])
    assert (a, tok) == (0, 2)
    r1 = p0[1] / (p0[1] + p0[2])
    assert gap == pytest.approx(min(0.5 - r1, 0.5), rel=1e-12)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_zero_temperature_limit_is_the_greedy_rule(seed):
    rng = np.random.default_rng(seed)
    M, V = 5, 1000
    z = rng.standard_normal((M, V))
    am = z.argmax(axis=1).astype(np.int32)
    for trial in range(20):
        hit = rng.random(M - 1) < 0.6
        draft = np.where(hit, am[:M - 1], rng.integers(0, V, M - 1)).astype(np.int32)
        a, tok, _, _ = oracle.spec_sample(z, 1e-9, draft, rng.random(M - 1), rng.random(M))
        assert (a, tok) == oracle.spec_verify(am, draft)


@pytest.mark.parametrize("T,draft", [(1.0, 3), (0.7, 0), (2.0, 5)])
def test_emitted_token_has_the_target_distribution(T, draft):
    """P(first emitted token = v) must equal softmax(z_0 / T)(v) for every v,
    whatever the drafted token: quadrature over a midpoint grid of the two
    uniforms that decide the first token."""
    rng = np.random.default_rng(7)
    V = 6
    z = rng.standard_normal((2, V)) * 1.5
    p = np.exp(z[0] / T - (z[0] / T).max())
    p /= p.sum()
    N = 300
    grid = (np.arange(N) + 0.5) / N
    counts = np.zeros(V)
    for ua in grid:
        for un in grid:
            a, tok, _, _ = oracle.spec_sample(z, T, [draft], [ua], [un, 0.5])
            counts[draft if a >= 1 else tok] += 1
    np.testing.assert_allclose(counts / N ** 2, p, atol=2.5 / N)


def test_single_position_is_an_inverse_cdf_sample():
    rng = np.random.default_rng(8)
    V, T = 500, 0.8
    z = rng.standard_normal((1, V)) * 3
    w = np.exp((z[0] - z[0].max()) / T)
    cdf = np.cumsum(w) / w.sum()
    for u in rng.random(200):
        a, tok, _, gap = oracle.spec_sample(z, T, [], [], [u])
        assert a == 0
        assert tok == int(np.searchsorted(cdf, u, side="right"))
        assert gap <= max(u - (cdf[tok - 1] if tok else 0.0), cdf[tok] - u) + 1e-12


def test_certain_draft_is_always_accepted():
    z = np.zeros((3, 50))
    z[0, 7] = 1e3
    z[1, 9] = 1e3
    a, tok, _, _ = oracle.spec_sample(z, 1.0, [7, 9], [0.999, 0.999], [0.3, 0.3, 0.3])
    assert a == 2 and tok == int(0.3 * 50)   # uniform last position: token floor(u V)


def test_logits_match_torch():
    emb = synth.embedding(51, vocab=777, hidden=64)
    h = bf16_values(synth.hidden_states(52, 3, hidden=64))
    z = oracle.lm_head_logits(bf16_bits(emb), h)
    ref = torch.from_numpy(h) @ emb.to(torch.float64).T
    np.testing.assert_allclose(z, ref.numpy(), rtol=1e-13, atol=1e-15)
