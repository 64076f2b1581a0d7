"""GPU parity of the MoE layer, the stack and the verify step with the
always-on 2816 x 2112 dense MLP in place of the shared expert ("llm-decoding"
§"Where the 7.36 GB goes") against the oracle's `fgmo_moe_layer_dense`, at
full size: 128 routed experts of the benchmark layers (Zipf bias) and
2112-wide E4M3 MLPs with fp32 row scales in their natural layout (down rows
2112 wide). Same rules as the layer test: router ids bit-exact where the
oracle's margin exceeds 1e-2 (else a valid choice), rows within 1e-2 and
elementwise within 2e-2 of the bf16-rounded oracle. The persistent kernel
(its down products on tcgen05 at M <= 5 on the default path, on mma.sync on
FGM_PATH_FUSED_MMA and at M > 5) and the per-stage kernels."""

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import (ELEM_TOL, MARGIN, REL_TOL, bf16_bits, bf16_values, elementwise_rel_err, id_sets_agree,
                     ids_valid_at_tie, rowwise_rel_err, to_oracle_layer)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", params=[0, 3, 1], ids=["fused", "fused_mma", "staged"])
def fgm(request):
    """fused: the persistent kernel with the MLP's three parts as its always-on
    slots (tcgen05 down products at M <= 5); fused_mma: the same with the
    mma.sync down products at every M; staged: the per-stage kernels."""
    import fine_grained_moe_gb300 as m
    m.lib()
    prev = m.select_path(request.param)
    yield m
    m.select_path(prev)


@pytest.fixture(scope="module")
def case():
    p = synth.layer(0, device="cuda", s=1.1)
    L = to_oracle_layer(p)
    d = synth.dense_mlp(7, device="cuda")
    D = oracle.MlpParams(**{k: v.cpu().numpy() for k, v in d.items()})
    return p, L, d, D


@pytest.mark.parametrize("M", [1, 5, 8])
def test_dense_layer_matches_oracle(fgm, case, M):
    p, L, d, D = case
    ws = fgm.Workspace("cuda")
    x = synth.hidden_states(3000 + M, M, device="cuda")
    ids = torch.empty((M, 8), dtype=torch.int32, device="cuda")
    y = fgm.moe_layer_dense_fwd(p, d, x, topk_ids=ids, ws=ws)
    torch.cuda.synchronize()
    ref = oracle.moe_layer(L, bf16_values(x), dense_shared=D)
    gid = ids.cpu().numpy()
    row, elem = rowwise_rel_err(y, ref.y), elementwise_rel_err(y, ref.y)
    compared = 0
    for t in range(M):
        if ref.margin[t] > MARGIN:
            assert id_sets_agree(gid[t], ref.ids[t]), (t, gid[t], ref.ids[t])
        else:
            assert ids_valid_at_tie(gid[t], ref.logits[t])
            if not id_sets_agree(gid[t], ref.ids[t]):
                continue
        assert row[t] <= REL_TOL, (t, row[t])
        assert elem[t] <= ELEM_TOL, (t, elem[t])
        compared += 1
    print(f"M={M}: {compared} tokens compared, row errors {np.round(row, 6).tolist()}")
    assert compared >= 1
    assert ws.status() == 0


def test_dense_layer_with_unaligned_down_scales(fgm, case):
    """The MLP's down-row scales 4 bytes off a 16-byte boundary (the ABI asks
    for 4-byte alignment): the tensor-memory down phase copies scales in
    16-byte units, so the call takes the mma.sync down products; the result
    still matches the oracle at M = 5."""
    p, L, d, D = case
    M = 5
    buf = torch.empty(d["down_s"].numel() + 1, dtype=torch.float32, device="cuda")
    buf[1:].copy_(d["down_s"].reshape(-1))
    d2 = dict(d)
    d2["down_s"] = buf[1:].view_as(d["down_s"])
    assert d2["down_s"].data_ptr() % 16 == 4
    ws = fgm.Workspace("cuda")
    x = synth.hidden_states(3000 + M, M, device="cuda")
    ids = torch.empty((M, 8), dtype=torch.int32, device="cuda")
    y = fgm.moe_layer_dense_fwd(p, d2, x, topk_ids=ids, ws=ws)
    torch.cuda.synchronize()
    ref = oracle.moe_layer(L, bf16_values(x), dense_shared=D)
    gid = ids.cpu().numpy()
    row, elem = rowwise_rel_err(y, ref.y), elementwise_rel_err(y, ref.y)
    compared = 0
    for t in range(M):
        if ref.margin[t] > MARGIN:
            assert id_sets_agree(gid[t], ref.ids[t]), (t, gid[t], ref.ids[t])
        elif not id_sets_agree(gid[t], ref.ids[t]):
            assert ids_valid_at_tie(gid[t], ref.logits[t])
            continue
        assert row[t] <= REL_TOL, (t, row[t])
        assert elem[t] <= ELEM_TOL, (t, elem[t])
        compared += 1
    assert compared >= 1
    assert ws.status() == 0


def test_dense_layer_is_routed_part_plus_mlp(fgm, case):
    """The dense call minus the plain layer call with the shared expert zeroed
    is the MLP alone (checked against the oracle's MLP per token)."""
    p, L, d, D = case
    ws = fgm.Workspace("cuda")
    M = 3
    x = synth.hidden_states(3100, M, device="cuda")
    q = dict(p)
    for k in ("gate_q", "up_q", "down_q"):
        q[k] = p[k].clone()
        q[k][128] = 0
    yd = fgm.moe_layer_dense_fwd(p, d, x, ws=ws).double()
    prev = fgm.select_path(fgm.PATH_STAGED)
    try:
        yr = fgm.moe_layer_fwd(q, x, ws=ws).double()
    finally:
        fgm.select_path(prev)
    xv = bf16_values(x)
    for t in range(M):
        mlp = oracle.mlp_token(D, xv[t])
        diff = (yd[t] - yr[t]).cpu().numpy()
        assert np.abs(diff - mlp).max() <= 2e-2 * np.abs(mlp).max() + 2 ** -7 * np.abs(yd[t].cpu().numpy()).max()


def test_dense_width_checked(fgm, case):
    p, _, d, _ = case
    x = synth.hidden_states(3200, 2, device="cuda")
    W = 700   # not a multiple of 704: rejected by the library's argument check
    bad = {"gate_q": d["gate_q"][:W].contiguous(), "gate_s": d["gate_s"][:W].contiguous(),
           "up_q": d["up_q"][:W].contiguous(), "up_s": d["up_s"][:W].contiguous(),
           "down_q": d["down_q"][:, :W].contiguous(), "down_s": d["down_s"]}
    with pytest.raises(fgm.FgmError):
        fgm.moe_layer_dense_fwd(p, bad, x)


# ------------------------------------------------------------------ stack and verify step
def _dense_stack_reference(host, mlps_host, h):
    """The oracle's stack with a dense MLP per layer: h <- h + layer(RMSNorm(h))
    (the decomposition `test_stack_layer_is_residual_of_normed_layer` pins),
    each layer the oracle's dense layer. Returns h and the trajectory."""
    traj = []
    for L, D in zip(host, mlps_host):
        out = oracle.moe_layer(L, oracle.rmsnorm(h), dense_shared=D)
        traj.append((out.ids.copy(), out.margin.copy(), h.copy()))
        h = h + out.y
    return h, traj


@pytest.mark.parametrize("n_layers,M", [(4, 5), (3, 8)])
def test_dense_stack_matches_oracle(fgm, n_layers, M):
    """A stack whose every layer carries a 2112-wide dense MLP in place of the
    shared expert (the persistent kernel with the MLP parts as always-on
    slots, or the per-stage kernels), per token against the oracle's stack:
    routing layer by layer (a first difference only at a near tie), final
    rows within 1e-2 for tokens that never diverge."""
    from test_gpu_parity import _compare_stack
    layers = [synth.layer(l + 1, device="cuda", s=1.1) for l in range(n_layers)]
    mlps = [synth.dense_mlp(20 + l, device="cuda") for l in range(n_layers)]
    ws = fgm.Workspace("cuda")
    x = synth.hidden_states(3300 + M, M, device="cuda")
    trace = torch.empty((n_layers, M, 8), dtype=torch.int32, device="cuda")
    y = fgm.moe_stack_dense_fwd(layers, mlps, x, ids_trace=trace, ws=ws)
    torch.cuda.synchronize()
    host = [to_oracle_layer(p) for p in layers]
    mlps_host = [oracle.MlpParams(**{k: v.cpu().numpy() for k, v in d.items()}) for d in mlps]
    h_ref, traj = _dense_stack_reference(host, mlps_host, bf16_values(x))
    full = _compare_stack(trace.cpu().numpy(), y, h_ref, traj, host, M)
    print(f"{n_layers} layers, M={M}: {len(full)} tokens compared to the end")
    assert len(full) >= 1
    assert ws.status() == 0


@pytest.fixture(scope="module")
def dense_verify_case():
    """30 benchmark layers, each with its own 2112-wide dense MLP, the
    262,144-word embedding, one input batch at M = 5 with drafts that copy the
    oracle's argmax with probability 0.7; the oracle's trajectory and argmax,
    one layer's host copy at a time."""
    n = 30
    layers = [synth.layer(l + 1, device="cuda", s=1.1) for l in range(n)]
    mlps = [synth.dense_mlp(40 + l, device="cuda") for l in range(n)]
    emb = synth.embedding(32, device="cuda")
    x = synth.hidden_states(3400, 5, device="cuda")
    h = bf16_values(x)
    traj, host = [], []
    for p, d in zip(layers, mlps):
        L = to_oracle_layer(p)
        D = oracle.MlpParams(**{k: v.cpu().numpy() for k, v in d.items()})
        out = oracle.moe_layer(L, oracle.rmsnorm(h), dense_shared=D)
        traj.append((out.ids.copy(), out.margin.copy(), h.copy()))
        host.append(L)
        h = h + out.y
    hn = oracle.bf16_to_f64(oracle.bf16_round(oracle.rmsnorm(h)))
    am, _, mg = oracle.lm_head(bf16_bits(emb), hn)
    draft = synth.drafts(35, am)
    return dict(layers=layers, mlps=mlps, emb=emb, x=x, h_ref=h, traj=traj, host=host, am=am, mg=mg,
                draft=draft)


def test_dense_verify_step_matches_oracle(fgm, dense_verify_case):
    """The full verify step (30 layers with dense MLPs, final norm, bf16
    lm_head, greedy accept): routing per layer, the argmax of every token whose
    trajectory matched the oracle and whose argmax margin exceeds 1e-2, and the
    accepted count and next token whenever the oracle's own accepted prefix is
    comparable."""
    from test_gpu_parity import _compare_stack
    c = dense_verify_case
    M = 5
    ws = fgm.Workspace("cuda")
    trace = torch.empty((30, M, 8), dtype=torch.int32, device="cuda")
    y = fgm.moe_stack_dense_fwd(c["layers"], c["mlps"], c["x"], ids_trace=trace, ws=ws)
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    out = fgm.verify_step_dense(c["layers"], c["mlps"], c["emb"], c["x"], c["draft"].cuda(), argmax=am, ws=ws)
    torch.cuda.synchronize()
    full = set(_compare_stack(trace.cpu().numpy(), y, c["h_ref"], c["traj"], c["host"], M))
    ok = [t in full and c["mg"][t] > MARGIN for t in range(M)]
    gam = am.cpu().numpy()
    for t in range(M):
        if ok[t]:
            assert gam[t] == c["am"][t], (t, gam[t], c["am"][t])
    a, nxt = out.cpu().tolist()
    assert (a, nxt) == oracle.spec_verify(gam, c["draft"].numpy())
    a_ref, nxt_ref = oracle.spec_verify(c["am"], c["draft"].numpy())
    if all(ok[:a_ref + 1]):
        assert (a, nxt) == (a_ref, nxt_ref)
    print(f"dense verify: {len(full)} tokens matched through 30 layers, comparable {ok}, accept {a, nxt}")
    assert sum(ok) >= 2
    assert ws.status() == 0
