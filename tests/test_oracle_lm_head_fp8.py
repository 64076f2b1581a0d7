"""Pins of the oracle's FP8 lm_head argmax.

Storing every weight in 8 bits, the tied output projection included, halves
the bytes a decode step streams ("llm-decoding", §"Lever 1: fewer bytes (FP8
weights)"; §"First principles: compute-bound or memory-bound?" puts that
projection at a fifth of a token's BF16 bytes). The rows are E4M3 codes with
one fp32 scale per row, the format of the expert weights, and a logit is the
row's scale times the dot product of its decoded codes with the hidden row.

The pins: a worked example computed by hand from the E4M3 definition; brute
force over fp64 logits from torch's float8 decode, with every finite code
present; equality with the bf16 lm_head where a power-of-two row scale makes
the dequantised rows exact bf16; one-hot hidden rows; ties; NaN codes.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import bf16_bits, bf16_values, dequant_torch


def test_worked_example_by_hand():
    # E4M3 codes by the format: 0x38 = +1.0 (exponent field 7), 0x40 = +2.0,
    # 0xB8 = -1.0, 0x01 = 1/8 * 2^-6 = 2^-9 (smallest subnormal)
    q = np.array([[0x38, 0x40], [0x40, 0xB8], [0x01, 0x38]], np.uint8)
    s = np.array([0.5, 1.0, 4.0], np.float32)
    h = np.array([[1.0, 1.0], [1.0, -1.0]])
    # token 0: 0.5 (1 + 2) = 1.5; 1 (2 - 1) = 1; 4 (2^-9 + 1) = 4.0078125
    # token 1: 0.5 (1 - 2) = -0.5; 1 (2 + 1) = 3; 4 (2^-9 - 1) = -3.9921875
    am, mx, mg = oracle.lm_head_fp8(q, s, h)
    assert am.tolist() == [2, 1]
    assert mx.tolist() == [4.0078125, 3.0]
    assert mg.tolist() == [4.0078125 - 1.5, 3.5]


@pytest.mark.parametrize("V,M", [(1000, 5), (777, 1), (4099, 8)])
def test_brute_force_against_torch_decode(V, M):
    rng = np.random.default_rng(V)
    H = 96
    q = rng.integers(0, 256, (V, H)).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x00                  # no NaN codes here
    q[0, :] = np.arange(H) % 0x7F                 # every finite code of either sign appears
    q[1, :] = (np.arange(H) + H) % 0x7F | 0x80
    s = (rng.random(V) * 1e-3 + 1e-5).astype(np.float32)
    h = bf16_values(synth.hidden_states(11, M, hidden=H))
    am, mx, mg = oracle.lm_head_fp8(q, s, h)
    z = torch.from_numpy(h) @ dequant_torch(q, s).T
    np.testing.assert_array_equal(am, torch.argmax(z, dim=1).numpy())
    np.testing.assert_allclose(mx, z.max(dim=1).values.numpy(), rtol=1e-12)
    top2 = torch.topk(z, 2, dim=1).values.numpy()
    np.testing.assert_allclose(mg, top2[:, 0] - top2[:, 1], rtol=1e-8, atol=1e-15)


def test_power_of_two_scales_equal_the_bf16_head():
    """With scale 2^-j every dequantised weight is an exact bf16 value, so the
    FP8 head must give the bf16 head's logits on those values, bit for bit."""
    emb = synth.embedding(21, vocab=2000, hidden=128)
    q, _ = synth.embedding_fp8(emb)
    j = torch.randint(4, 12, (2000,), generator=torch.Generator().manual_seed(3))
    s = torch.pow(2.0, -j.to(torch.float64)).to(torch.float32)
    deq = q.view(torch.float8_e4m3fn).to(torch.float64) * s.to(torch.float64).unsqueeze(1)
    deq_bf16 = deq.to(torch.bfloat16)
    assert torch.equal(deq_bf16.to(torch.float64), deq)          # exact in bf16
    h = bf16_values(synth.hidden_states(22, 6, hidden=128))
    a8, m8, g8 = oracle.lm_head_fp8(q.numpy(), s.numpy(), h)
    a16, m16, g16 = oracle.lm_head(bf16_bits(deq_bf16), h)
    np.testing.assert_array_equal(a8, a16)
    np.testing.assert_array_equal(m8, m16)
    np.testing.assert_array_equal(g8, g16)


def test_one_hot_hidden_reads_one_scaled_column():
    emb = synth.embedding(23, vocab=513, hidden=40)
    q, s = synth.embedding_fp8(emb)
    h = np.zeros((1, 40))
    h[0, 9] = 1.0
    am, mx, _ = oracle.lm_head_fp8(q.numpy(), s.numpy(), h)
    col = dequant_torch(q.numpy(), s.numpy())[:, 9].numpy()
    assert am[0] == int(np.argmax(col)) and mx[0] == col.max()


def test_ties_go_to_lower_index():
    emb = synth.embedding(24, vocab=300, hidden=32)
    q, s = synth.embedding_fp8(emb)
    q[250], s[250] = q[17], s[17]
    q[299], s[299] = q[17], s[17]
    h = dequant_torch(q[17:18].numpy(), s[17:18].numpy()).numpy() * 10.0
    am, _, mg = oracle.lm_head_fp8(q.numpy(), s.numpy(), h)
    assert am[0] == 17 and mg[0] == 0.0


def test_nan_code_rows_never_win():
    emb = synth.embedding(25, vocab=400, hidden=64)
    q, s = synth.embedding_fp8(emb)
    h = bf16_values(synth.hidden_states(26, 2, hidden=64))
    am0, mx0, _ = oracle.lm_head_fp8(q.numpy(), s.numpy(), h)
    q[am0[0], 5] = 0x7F                           # S.1111.111 is NaN
    am1, mx1, _ = oracle.lm_head_fp8(q.numpy(), s.numpy(), h)
    z = torch.from_numpy(h) @ dequant_torch(q.numpy(), s.numpy()).T
    z[:, am0[0]] = -np.inf
    assert am1[0] != am0[0]
    np.testing.assert_array_equal(am1, torch.argmax(z, dim=1).numpy())


def test_embedding_quantiser_matches_the_oracle_quantiser():
    emb = synth.embedding(27, vocab=257, hidden=64)
    q, s = synth.embedding_fp8(emb, chunk_rows=100)
    rq, rs = oracle.quantize_rows(emb.to(torch.float32).numpy())
    np.testing.assert_array_equal(q.numpy(), rq)
    np.testing.assert_array_equal(s.numpy(), rs)
