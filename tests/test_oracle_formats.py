"""Pins of the oracle's number formats (E4M3, bf16) and elementwise pieces.

The pages store weights in 8 bits and dequantise them at higher precision
("llm-decoding", §"Lever 1: fewer bytes (FP8 weights)"); the format is the
OCP FP8 E4M3 ("fn") encoding named by the benchmark configuration. These tests
pin the oracle's formula decode and brute-force encoder to values fixed by the
format itself and to torch's float8 conversion as an independent library.
"""

import math

import numpy as np
import pytest
import torch

import oracle


def test_e4m3_known_codes():
    # Values fixed by the format: bias 7, 3 mantissa bits, subnormal step 2^-9.
    table = {
        0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
        0x38: 1.0, 0x39: 1.125, 0x40: 2.0, 0x7E: 448.0, 0x77: 240.0,
        0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0,
    }
    codes = np.array(list(table), np.uint8)
    got = oracle.e4m3_decode(codes)
    for c, v in zip(codes, got):
        assert v == table[int(c)], hex(c)
    assert math.copysign(1.0, oracle.e4m3_decode(np.array([0x80], np.uint8))[0]) == -1.0
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(lib)
    assert (np.isnan(ours) == nan).all()
    assert nan.sum() == 2
    np.testing.assert_array_equal(ours[~nan], lib[~nan])


def test_e4m3_decode_monotone_and_symmetric():
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert (np.diff(pos) > 0).all()
    neg = oracle.e4m3_decode(np.arange(0x80, 0xFF, dtype=np.uint8))
    np.testing.assert_array_equal(neg, -pos)


def test_e4m3_encode_roundtrip_exact():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode(codes)
    back = oracle.e4m3_encode(vals)
    np.testing.assert_array_equal(back, codes)


def test_e4m3_encode_ties_to_even_and_saturation():
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2.0
    codes = oracle.e4m3_encode(mids)
    # a midpoint goes to whichever neighbour has an even code
    lower = np.arange(0x7E, dtype=np.uint8)
    expect = np.where(lower % 2 == 0, lower, lower + 1).astype(np.uint8)
    np.testing.assert_array_equal(codes, expect)
    big = oracle.e4m3_encode(np.array([448.0, 460.0, 1e6, -1e6, -449.0]))
    np.testing.assert_array_equal(big, np.array([0x7E, 0x7E, 0x7E, 0xFE, 0xFE], np.uint8))


def test_e4m3_encode_matches_torch_cast():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1.0, 30.0, 300.0)])
    v = np.clip(v, -448, 448).astype(np.float32)
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2.0).astype(np.float32)
    v = np.concatenate([v, mids, -mids])
    ours = oracle.e4m3_encode(v.astype(np.float64))
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, lib)
    assert not np.isin(ours, [0x7F, 0xFF]).any()


def test_quantize_rows_matches_input_recipe():
    """The oracle's per-row quantiser and the input generator's torch cast agree."""
    import synth
    g = torch.Generator().manual_seed(3)
    w = torch.randn((37, 160), generator=g) * 0.02
    w[5] = 0.0
    q_t, s_t = synth.quantize_rows_e4m3(w)
    q_o, s_o = oracle.quantize_rows(w.numpy())
    np.testing.assert_array_equal(s_o, s_t.numpy())
    np.testing.assert_array_equal(q_o, q_t.numpy())
    assert s_o[5] == 1.0 and (q_o[5] == 0).all()
    # the largest magnitude of each non-zero row lands on the top code
    amax_code = (q_o & 0x7F).max(axis=1)
    assert (amax_code[np.arange(37) != 5] == 0x7E).all()


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(50000) * s for s in (1e-30, 1e-3, 1.0, 1e5)])
    v32 = v.astype(np.float32)
    ours = oracle.bf16_round(v32.astype(np.float64))
    lib = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, lib)
    # exact ties: halfway between two bf16 neighbours goes to the even one
    base = np.array([1.0, 1.0 + 2 ** -7, 3.0, 1000.0], np.float64)
    ulp = np.array([2 ** -7, 2 ** -7, 2 ** -6, 4.0])
    ties = oracle.bf16_round(base + ulp / 2)
    lib_t = torch.tensor(base + ulp / 2, dtype=torch.float64).to(torch.float32).to(torch.bfloat16)
    np.testing.assert_array_equal(ties, lib_t.view(torch.int16).numpy().view(np.uint16))
    back = oracle.bf16_to_f64(ours)
    assert np.all(np.abs(back - v32) <= np.abs(v32) * 2.0 ** -8 + 1e-45)


def test_gelu_tanh_against_torch_and_identities():
    x = np.linspace(-12, 12, 4001)
    ours = oracle.gelu_tanh(x)
    lib = torch.nn.functional.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    np.testing.assert_allclose(ours, lib, rtol=1e-13, atol=1e-14)
    # closed forms: gelu(0) = 0; gelu(x) - gelu(-x) = x; tends to x and 0 at the tails
    assert oracle.gelu_tanh(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(ours - oracle.gelu_tanh(-x), x, rtol=0, atol=1e-12)
    assert abs(oracle.gelu_tanh(np.array([30.0]))[0] - 30.0) < 1e-12
    assert abs(oracle.gelu_tanh(np.array([-30.0]))[0]) < 1e-12


def test_rmsnorm_closed_forms():
    rng = np.random.default_rng(2)
    h = rng.standard_normal((3, 512)) * np.array([[0.1], [1.0], [25.0]])
    out = oracle.rmsnorm(h, eps=0.0)
    np.testing.assert_allclose(np.sqrt((out ** 2).mean(axis=1)), 1.0, rtol=1e-13)
    np.testing.assert_allclose(oracle.rmsnorm(7.0 * h, eps=0.0), out, rtol=1e-13)
    # constant row c: c / sqrt(c^2 + eps)
    c = np.full((1, 64), 0.5)
    np.testing.assert_allclose(oracle.rmsnorm(c, eps=1e-6), 0.5 / math.sqrt(0.25 + 1e-6), rtol=1e-14)
    assert (oracle.rmsnorm(np.zeros((1, 8)), eps=1e-6) == 0).all()
