"""Pins of the oracle's lm_head argmax and greedy acceptance.

The tied 262,144-word lm_head is read once per step ("llm-decoding",
§"Where the 7.36 GB goes"); the target verifies the drafted tokens in one pass
and keeps the ones it would have produced itself (§"Lever 2: fewer passes
(native MTP)"), which at temperature 0 is the longest draft prefix equal to
the target's own argmax tokens, followed by the target's token at the first
mismatch. The pins: brute-force argmax over fp64 logits from torch's bf16
decode, explicit ties, and every hit/miss pattern of the drafts.
"""

import itertools

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import bf16_bits, bf16_values


@pytest.mark.parametrize("V,M", [(1000, 5), (777, 1), (4099, 8)])
def test_lm_head_argmax_brute_force(V, M):
    emb = synth.embedding(5, vocab=V, hidden=96)
    h = bf16_values(synth.hidden_states(6, M, hidden=96))
    am, mx, mg = oracle.lm_head(bf16_bits(emb), h)
    z = torch.from_numpy(h) @ emb.to(torch.float64).T
    np.testing.assert_array_equal(am, torch.argmax(z, dim=1).numpy())
    np.testing.assert_allclose(mx, z.max(dim=1).values.numpy(), rtol=1e-13)
    top2 = torch.topk(z, 2, dim=1).values.numpy()
    np.testing.assert_allclose(mg, top2[:, 0] - top2[:, 1], rtol=1e-9, atol=1e-13)


def test_lm_head_ties_go_to_lower_index():
    emb = synth.embedding(7, vocab=300, hidden=32)
    emb[250] = emb[17]
    emb[299] = emb[17]
    h = emb[17:18].to(torch.float64).numpy() * 10.0   # row 17 (and its copies) wins
    am, mx, mg = oracle.lm_head(bf16_bits(emb), h)
    assert am[0] == 17 and mg[0] == 0.0


def test_lm_head_one_hot_hidden_reads_one_column():
    emb = synth.embedding(8, vocab=513, hidden=40)
    h = np.zeros((1, 40))
    h[0, 9] = 1.0
    am, mx, _ = oracle.lm_head(bf16_bits(emb), h)
    col = bf16_values(emb)[:, 9]
    assert am[0] == int(np.argmax(col)) and mx[0] == col.max()


@pytest.mark.parametrize("gamma", range(0, 8))
def test_accept_length_every_pattern(gamma):
    rng = np.random.default_rng(gamma)
    target = rng.integers(0, 1000, gamma + 1).astype(np.int32)
    for pattern in itertools.product((True, False), repeat=gamma):
        draft = np.array([target[i] if hit else (target[i] + 1 + i) % 1000
                          for i, hit in enumerate(pattern)], np.int32)
        a, nxt = oracle.spec_verify(target, draft)
        lead = 0
        for hit in pattern:
            if not hit:
                break
            lead += 1
        assert a == lead and nxt == target[lead]


def test_accept_special_cases():
    t = np.array([4, 9, 9, 2, 7], np.int32)
    assert oracle.spec_verify(t, np.array([5, 9, 9, 2], np.int32)) == (0, 4)   # first draft wrong
    assert oracle.spec_verify(t, np.array([4, 9, 9, 2], np.int32)) == (4, 7)   # all accepted
    assert oracle.spec_verify(t, np.array([4, 9, 3, 2], np.int32)) == (2, 9)   # later hits ignored
    assert oracle.spec_verify(np.array([3], np.int32), np.zeros(0, np.int32)) == (0, 3)


def test_draft_recipe_acceptance_rate():
    """Drafts that copy the target with p = 0.7 give E[a] = 0.7 + 0.7^2 + 0.7^3 + 0.7^4."""
    acc = []
    for s in range(4000):
        t = np.arange(5, dtype=np.int32) + 10 * s
        d = synth.drafts(s, t, vocab=1 << 30).numpy()
        acc.append(oracle.spec_verify(t, d)[0])
    expect = sum(0.7 ** j for j in range(1, 5))
    assert abs(np.mean(acc) - expect) < 0.06
