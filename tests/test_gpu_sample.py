"""GPU parity of speculative sampling at temperature T > 0 against the oracle.

The CUDA call returns the logits z it computed and {accepted drafts, emitted
token}; the oracle takes its own fp64 logits of the same bf16 embedding and
hidden rows, the same drafts (which copy the oracle's argmax with probability
0.7) and the same fp32 uniforms. Rules:
  * logits within 1e-2 relative of the oracle's (row infinity norm), and in
    fact within 1e-4 of the row's largest magnitude;
  * accepted count and token identical wherever the oracle's decision margins
    exceed SAMPLE_TOL(T): |u_acc - p(d)| and the inverse-CDF gap relative to
    the distribution's mass. The GPU's logits differ from the oracle's by up
    to ~1e-5 (fp32 accumulation of 2816 products), which moves every weight
    exp((z - max) / T) by a relative 1e-5 / T, so decisions closer than that
    may go either way; SAMPLE_TOL(T) = 2e-4 / T leaves 20x room;
  * every emitted token, compared or not, lies where the oracle's fp64 CDF of
    the emitting position puts the target, up to the same tolerance.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import REL_TOL, bf16_bits, bf16_values, rowwise_rel_err

pytestmark = pytest.mark.gpu


def sample_tol(T: float) -> float:
    return 2e-4 / T


@pytest.fixture(scope="module")
def fgm():
    import fine_grained_moe_gb300 as m
    m.lib()
    return m


@pytest.fixture(scope="module")
def ws(fgm):
    return fgm.Workspace("cuda")


def _cdf_brackets(z_ref, T, a, tok, draft, u_next, tol):
    """The emitted token is the inverse-CDF sample of the oracle's fp64 weights
    at position a (the draft of a rejected position removed), up to tol."""
    M = z_ref.shape[0]
    w = np.exp((z_ref[a] - z_ref[a].max()) / T)
    if a < M - 1:
        w[draft[a]] = 0.0
    c = np.cumsum(w)
    target = float(u_next[a]) * c[-1]
    lo = c[tok - 1] if tok > 0 else 0.0
    assert w[tok] > 0.0, (a, tok)
    assert lo - tol * c[-1] <= target <= c[tok] + tol * c[-1], (a, tok, lo / c[-1], target / c[-1], c[tok] / c[-1])


def _run_case(fgm, ws, emb, h, T, seed, trials):
    M = h.shape[0]
    z_ref = oracle.lm_head_logits(bf16_bits(emb), bf16_values(h))
    am_ref = z_ref.argmax(axis=1).astype(np.int32)
    draft = synth.drafts(seed, am_ref, vocab=emb.shape[0])
    tol = sample_tol(T)
    compared = 0
    for k in range(trials):
        u_acc = synth.uniforms(1000 * seed + 2 * k, M - 1)
        u_next = synth.uniforms(1000 * seed + 2 * k + 1, M)
        am = torch.empty(M, dtype=torch.int32, device="cuda")
        out, z = fgm.lm_head_sample(emb, h, T, draft.cuda() if M > 1 else None, u_acc.cuda() if M > 1 else None,
                                    u_next.cuda(), argmax=am, ws=ws)
        torch.cuda.synchronize()
        a, tok = out.cpu().tolist()
        if k == 0:
            zg = z.cpu().double().numpy()
            assert (rowwise_rel_err(z.to(torch.bfloat16), z_ref) <= REL_TOL).all()
            assert (np.abs(zg - z_ref).max(axis=1) <= 1e-4 * np.abs(z_ref).max(axis=1)).all()
        a_ref, tok_ref, mg, gap = oracle.spec_sample(z_ref, T, draft.numpy(), u_acc.double().numpy(),
                                                     u_next.double().numpy())
        assert 0 <= a <= M - 1 and 0 <= tok < emb.shape[0], (a, tok)
        if mg > tol:
            assert a == a_ref, (T, k, a, a_ref, mg)
            _cdf_brackets(z_ref, T, a, tok, draft.numpy(), u_next.numpy(), tol)
            if gap > tol:
                assert tok == tok_ref, (T, k, tok, tok_ref, gap)
                compared += 1
    assert ws.status() == 0
    return compared


@pytest.mark.parametrize("V,M", [(4099, 5), (50021, 8), (50021, 1), (262144, 5), (7, 3)])
@pytest.mark.parametrize("T", [0.02, 0.1, 0.3, 1.0])
def test_lm_head_sample_matches_oracle(fgm, ws, V, M, T):
    emb = synth.embedding(32, vocab=V, device="cuda")
    h = synth.hidden_states(2000 + M, M, device="cuda")
    compared = _run_case(fgm, ws, emb, h, T, seed=3 + M, trials=8)
    print(f"V={V} M={M} T={T}: {compared} of 8 trials compared exactly")
    if T <= 0.3 or V <= 7:
        assert compared >= 2


def test_zero_temperature_limit_is_greedy(fgm, ws):
    """T = 1e-4: every weight but the maximum's underflows, so the sampling
    verify is greedy acceptance on the argmax."""
    V, M = 50021, 6
    emb = synth.embedding(32, vocab=V, device="cuda")
    h = synth.hidden_states(2100, M, device="cuda")
    am_gpu = fgm.lm_head_argmax(emb, h, ws=ws).cpu().numpy()
    for k in range(6):
        draft = synth.drafts(50 + k, am_gpu, vocab=V)
        out, _ = fgm.lm_head_sample(emb, h, 1e-4, draft.cuda(), synth.uniforms(60 + k, M - 1).cuda(),
                                    synth.uniforms(70 + k, M).cuda(), ws=ws)
        assert tuple(out.cpu().tolist()) == oracle.spec_verify(am_gpu, draft.numpy())
    assert ws.status() == 0


def test_sample_rejects_bad_temperature(fgm, ws):
    emb = synth.embedding(32, vocab=64, device="cuda")
    h = synth.hidden_states(2200, 2, device="cuda")
    d = torch.zeros(1, dtype=torch.int32, device="cuda")
    u = torch.zeros(2, dtype=torch.float32, device="cuda")
    for T in (0.0, -1.0, float("inf"), float("nan"), 1e-39):
        with pytest.raises(fgm.FgmError):
            fgm.lm_head_sample(emb, h, T, d, u[:1], u, ws=ws)
