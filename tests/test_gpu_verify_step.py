"""GPU parity of the full-size stack and verify step against the oracle.

Thirty layers of the M = 5 Zipf(1.1) configuration (per-layer seeds 1..30,
about 23 GB of E4M3 expert weights), the final unit RMSNorm rounded to bf16,
the 262,144-word tied lm_head and greedy acceptance of four drafts that copy
the oracle's argmax with probability 0.7. The oracle runs layer by layer on
host copies of the same weights.
"""

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import MARGIN, REL_TOL, bf16_bits, bf16_values, rowwise_rel_err, to_oracle_layer
from test_gpu_parity import _compare_stack

pytestmark = pytest.mark.gpu

M = 5
N_LAYERS = 30


@pytest.fixture(scope="module", params=[0, 1], ids=["fused", "staged"])
def setup(request):
    import fine_grained_moe_gb300 as fgm
    fgm.lib()
    prev = fgm.select_path(request.param)
    layers = [synth.layer(l + 1, device="cuda", s=1.1) for l in range(N_LAYERS)]
    emb = synth.embedding(32, device="cuda")
    x = synth.hidden_states(31, M, device="cuda")
    # oracle trajectory, one layer's host copy at a time
    h = bf16_values(x)
    traj, host = [], []
    for p in layers:
        L = to_oracle_layer(p)
        out = oracle.stack_layer(L, h)
        traj.append((out.ids.copy(), out.margin.copy(), h.copy()))
        host.append(L)
        h = out.y
    hn_bits = oracle.bf16_round(oracle.rmsnorm(h))
    am, mx, mg = oracle.lm_head(bf16_bits(emb), oracle.bf16_to_f64(hn_bits))
    draft = synth.drafts(33, am)
    yield dict(fgm=fgm, layers=layers, emb=emb, x=x, h_ref=h, traj=traj, host=host, am=am, mg=mg,
               draft=draft, hn=oracle.bf16_to_f64(hn_bits), ws=fgm.Workspace("cuda"))
    fgm.select_path(prev)


def test_stack_30_layers(setup):
    s = setup
    trace = torch.empty((N_LAYERS, M, 8), dtype=torch.int32, device="cuda")
    y = s["fgm"].moe_stack_fwd(s["layers"], s["x"], ids_trace=trace, ws=s["ws"])
    torch.cuda.synchronize()
    full = _compare_stack(trace.cpu().numpy(), y, s["h_ref"], s["traj"], s["host"], M)
    assert len(full) >= 2, full
    assert s["ws"].status() == 0


def _matched_positions(s):
    """Positions whose routing matched the oracle's in every layer."""
    trace = torch.empty((N_LAYERS, M, 8), dtype=torch.int32, device="cuda")
    y = s["fgm"].moe_stack_fwd(s["layers"], s["x"], ids_trace=trace, ws=s["ws"])
    torch.cuda.synchronize()
    return set(_compare_stack(trace.cpu().numpy(), y, s["h_ref"], s["traj"], s["host"], M))


def _comparable_prefix(s, margins=None):
    """Positions whose whole trajectory matched the oracle and whose argmax is
    decided by more than the margin (the bf16 head's unless given)."""
    full = _matched_positions(s)
    mg = s["mg"] if margins is None else margins
    return [t in full and mg[t] > MARGIN for t in range(M)]


def test_verify_step_accept_and_next(setup):
    s = setup
    fgm = s["fgm"]
    draft = s["draft"].cuda()
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    out = fgm.verify_step(s["layers"], s["emb"], s["x"], draft, argmax=am, ws=s["ws"])
    torch.cuda.synchronize()
    a_ref, nxt_ref = oracle.spec_verify(s["am"], s["draft"].numpy())
    ok = _comparable_prefix(s)
    gam = am.cpu().numpy()
    for t in range(M):
        if ok[t]:
            assert gam[t] == s["am"][t], (t, gam[t], s["am"][t])
    a, nxt = out.cpu().tolist()
    # the accept rule applied to the GPU's own argmax is always exact
    assert (a, nxt) == oracle.spec_verify(gam, s["draft"].numpy())
    if all(ok[:a_ref + 1]):
        assert (a, nxt) == (a_ref, nxt_ref)
    assert s["ws"].status() == 0


def test_verify_step_host_buffers_match(setup):
    s = setup
    fgm = s["fgm"]
    out_dev = fgm.verify_step(s["layers"], s["emb"], s["x"], s["draft"].cuda(), ws=s["ws"])
    x_h = s["x"].cpu().pin_memory()
    d_h = s["draft"].clone().pin_memory()
    out_h = torch.empty(2, dtype=torch.int32).pin_memory()
    fgm.verify_step_host(s["layers"], s["emb"], x_h, d_h, out_host=out_h, ws=s["ws"])
    assert out_h.tolist() == out_dev.cpu().tolist()


def test_verify_step_m1_no_drafts(setup):
    s = setup
    fgm = s["fgm"]
    x1 = s["x"][:1].contiguous()
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    out = fgm.verify_step(s["layers"], s["emb"], x1, None, argmax=am, ws=s["ws"])
    assert out.cpu().tolist() == [0, int(am.cpu()[0])]
    # batch invariance: token 0 alone reaches the same argmax as inside M = 5
    am5 = torch.empty(M, dtype=torch.int32, device="cuda")
    fgm.verify_step(s["layers"], s["emb"], s["x"], s["draft"].cuda(), argmax=am5, ws=s["ws"])
    if s["mg"][0] > MARGIN:
        assert int(am.cpu()[0]) == int(am5.cpu()[0])


def test_stack_and_verify_m8(setup):
    """M = 8 (gamma = 7) runs the three-block packing of the persistent kernel;
    full size, against the oracle trajectory of the same 30 layers."""
    s = setup
    fgm = s["fgm"]
    m = 8
    x = synth.hidden_states(41, m, device="cuda")
    h = bf16_values(x)
    traj = []
    for L in s["host"]:
        out = oracle.stack_layer(L, h)
        traj.append((out.ids.copy(), out.margin.copy(), h.copy()))
        h = out.y
    trace = torch.empty((N_LAYERS, m, 8), dtype=torch.int32, device="cuda")
    y = fgm.moe_stack_fwd(s["layers"], x, ids_trace=trace, ws=s["ws"])
    torch.cuda.synchronize()
    full = _compare_stack(trace.cpu().numpy(), y, h, traj, s["host"], m)
    assert len(full) >= 2, full
    hn_bits = oracle.bf16_round(oracle.rmsnorm(h))
    am_ref, _, mg = oracle.lm_head(bf16_bits(s["emb"]), oracle.bf16_to_f64(hn_bits))
    draft = synth.drafts(43, am_ref)
    am = torch.empty(m, dtype=torch.int32, device="cuda")
    out = fgm.verify_step(s["layers"], s["emb"], x, draft.cuda(), argmax=am, ws=s["ws"])
    torch.cuda.synchronize()
    gam = am.cpu().numpy()
    for t in full:
        if mg[t] > MARGIN:
            assert gam[t] == am_ref[t], (t, gam[t], am_ref[t])
    assert tuple(out.cpu().tolist()) == oracle.spec_verify(gam, draft.numpy())
    assert s["ws"].status() == 0


def test_verify_step_fp8_head(setup):
    """The same step with the FP8 lm_head: the embedding's E4M3 copy read by
    the FP8 kernel, against the oracle's FP8 head on the oracle's own final
    normed hidden rows; drafts copy that head's argmax with probability 0.7."""
    s = setup
    fgm = s["fgm"]
    q, sc = synth.embedding_fp8(s["emb"])
    am_ref, _, mg_ref = oracle.lm_head_fp8(q.cpu().numpy(), sc.cpu().numpy(), s["hn"])
    draft = synth.drafts(34, am_ref)
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    out = fgm.verify_step_fp8_head(s["layers"], q, sc, s["x"], draft.cuda(), argmax=am, ws=s["ws"])
    torch.cuda.synchronize()
    ok = _comparable_prefix(s, mg_ref)
    gam = am.cpu().numpy()
    for t in range(M):
        if ok[t]:
            assert gam[t] == am_ref[t], (t, gam[t], am_ref[t])
    a, nxt = out.cpu().tolist()
    assert (a, nxt) == oracle.spec_verify(gam, draft.numpy())
    a_ref, nxt_ref = oracle.spec_verify(am_ref, draft.numpy())
    if all(ok[:a_ref + 1]):
        assert (a, nxt) == (a_ref, nxt_ref)
    assert s["ws"].status() == 0


def test_verify_step_fp8_head_m1(setup):
    """M = 1 through the FP8 head: no drafts, the next token is the argmax."""
    s = setup
    fgm = s["fgm"]
    q, sc = synth.embedding_fp8(s["emb"])
    x1 = s["x"][:1].contiguous()
    am = torch.empty(1, dtype=torch.int32, device="cuda")
    out = fgm.verify_step_fp8_head(s["layers"], q, sc, x1, None, argmax=am, ws=s["ws"])
    assert out.cpu().tolist() == [0, int(am.cpu()[0])]
    assert s["ws"].status() == 0
