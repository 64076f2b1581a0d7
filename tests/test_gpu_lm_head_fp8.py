"""GPU parity of the FP8 lm_head (E4M3 embedding rows with fp32 row scales)
against the oracle: argmax bit-exact where the oracle's top-1/top-2 margin
exceeds 1e-2, otherwise the chosen row's oracle logit within 1e-2 of the top;
the winning logit within 1e-4. Sizes from one ragged tile to the full
262,144-word vocabulary; the edge cases are ties, NaN codes and hidden rows of
extreme magnitude (the power-of-two scaling of the hidden rows' E4M3 terms).
Both kernels: the mma.sync one and the tensor-memory one (tcgen05)."""

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import MARGIN, bf16_values, dequant_torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=[0, 1, 2], ids=["fused", "staged", "fused_tc"])
def fgm(request):
    """fused and staged: the mma.sync kernel; fused_tc: the tensor-memory kernel
    (tcgen05.mma, TMA tensor copies)."""
    import fine_grained_moe_gb300 as m
    m.lib()
    prev = m.select_path(request.param)
    yield m
    m.select_path(prev)


@pytest.fixture(scope="module")
def ws(fgm):
    return fgm.Workspace("cuda")


def _fp8(seed, V):
    emb = synth.embedding(seed, vocab=V, device="cuda")
    q, s = synth.embedding_fp8(emb)
    del emb
    return q, s


def _check(q, s, h, am, mx):
    qh, sh = q.cpu().numpy(), s.cpu().numpy()
    hv = bf16_values(h)
    ram, rmx, rmg = oracle.lm_head_fp8(qh, sh, hv)
    gam = am.cpu().numpy()
    for t in range(h.shape[0]):
        if rmg[t] > MARGIN:
            assert gam[t] == ram[t], (t, gam[t], ram[t], rmg[t])
        else:
            z = float(dequant_torch(qh[gam[t]:gam[t] + 1], sh[gam[t]:gam[t] + 1])[0].numpy() @ hv[t])
            assert z >= rmx[t] - MARGIN
    np.testing.assert_allclose(mx.cpu().numpy(), rmx, rtol=1e-4, atol=1e-4)
    return ram, rmx


@pytest.mark.parametrize("V,M", [(262144, 5), (50021, 1), (50021, 8), (1, 3), (17, 2), (4099, 6)])
def test_lm_head_fp8_matches_oracle(fgm, ws, V, M):
    q, s = _fp8(32, V)
    h = synth.hidden_states(31, M, device="cuda")
    mx = torch.empty(M, dtype=torch.float32, device="cuda")
    am = fgm.lm_head_argmax_fp8(q, s, h, maxlogit=mx, ws=ws)
    torch.cuda.synchronize()
    _check(q, s, h, am, mx)
    assert ws.status() == 0


def test_lm_head_fp8_ties_to_lower_index(fgm, ws):
    q, s = _fp8(9, 5000)
    for r in (4321, 4999):
        q[r] = q[77]
        s[r] = s[77]
    deq = (q[77].view(torch.float8_e4m3fn).float() * s[77]).to(torch.bfloat16)
    h = deq.unsqueeze(0).repeat(2, 1).contiguous()
    am = fgm.lm_head_argmax_fp8(q, s, h, ws=ws)
    assert am.cpu().tolist() == [77, 77]


@pytest.mark.parametrize("e", [40, -60, 100])
def test_lm_head_fp8_extreme_hidden_magnitudes(fgm, ws, e):
    """h * 2^e is exact in bf16; the argmax must not move and the winning logit
    must scale by 2^e, although h * 2^40 overflows f16 and h * 2^-60 underflows
    it without the kernel's per-token scaling."""
    q, s = _fp8(12, 30011)
    h = synth.hidden_states(13, 4, device="cuda")
    hs = (h.float() * 2.0 ** e).to(torch.bfloat16)
    assert torch.equal(hs.float() * 2.0 ** -e, h.float())
    mx0 = torch.empty(4, dtype=torch.float32, device="cuda")
    mx1 = torch.empty(4, dtype=torch.float32, device="cuda")
    am0 = fgm.lm_head_argmax_fp8(q, s, h, maxlogit=mx0, ws=ws)
    am1 = fgm.lm_head_argmax_fp8(q, s, hs, maxlogit=mx1, ws=ws)
    torch.cuda.synchronize()
    assert am0.cpu().tolist() == am1.cpu().tolist()
    np.testing.assert_allclose(mx1.cpu().double().numpy() * 2.0 ** -e, mx0.cpu().double().numpy(), rtol=1e-6)
    _check(q, s, hs, am1, mx1)


def test_lm_head_fp8_nan_code_row_never_wins(fgm, ws):
    q, s = _fp8(14, 20011)
    h = synth.hidden_states(15, 3, device="cuda")
    am0 = fgm.lm_head_argmax_fp8(q, s, h, ws=ws)
    q[int(am0[0])][100] = 0x7F
    mx = torch.empty(3, dtype=torch.float32, device="cuda")
    am1 = fgm.lm_head_argmax_fp8(q, s, h, maxlogit=mx, ws=ws)
    torch.cuda.synchronize()
    assert int(am1[0]) != int(am0[0])
    _check(q, s, h, am1, mx)
    assert ws.status() == 0


def test_lm_head_fp8_agrees_with_bf16_head_on_exact_rows(fgm, ws):
    """Rows whose dequantised values are exact bf16 (power-of-two scales): the
    FP8 and bf16 kernels read the same matrix and must pick the same rows."""
    q, _ = _fp8(16, 40009)
    j = torch.randint(4, 12, (40009,), device="cuda", generator=torch.Generator("cuda").manual_seed(5))
    s = torch.pow(2.0, -j.float())
    emb = (q.view(torch.float8_e4m3fn).float() * s.unsqueeze(1)).to(torch.bfloat16)
    h = synth.hidden_states(17, 7, device="cuda")
    m8 = torch.empty(7, dtype=torch.float32, device="cuda")
    m16 = torch.empty(7, dtype=torch.float32, device="cuda")
    a8 = fgm.lm_head_argmax_fp8(q, s, h, maxlogit=m8, ws=ws)
    a16 = fgm.lm_head_argmax(emb, h, maxlogit=m16, ws=ws)
    torch.cuda.synchronize()
    _, _, rmg = oracle.lm_head_fp8(q.cpu().numpy(), s.cpu().numpy(), bf16_values(h))
    for t in range(7):
        if rmg[t] > MARGIN:
            assert int(a8[t]) == int(a16[t])
    np.testing.assert_allclose(m8.cpu().numpy(), m16.cpu().numpy(), rtol=1e-5, atol=1e-5)
