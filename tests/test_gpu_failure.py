"""Failure detection on the GPU without a fault. Every wait inside the
persistent kernel has a time limit. A test hook makes the next launch wait on
a grid barrier that no CTA can complete (a flag that nothing sets); the wait
must run out within the limit, the kernel must raise the timeout status bit
and exit, and the same context and workspace must then give correct results.
"""

import time

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def test_unreachable_barrier_times_out_then_recovers():
    import fine_grained_moe_gb300 as m
    prev_path = m.select_path(m.PATH_FUSED)
    prev_limit = m.set_wait_limit_ns(50_000_000)   # 50 ms
    try:
        ws = m.Workspace("cuda")
        p = synth.layer(0, device="cuda", s=1.1)
        x = synth.hidden_states(5, 3, device="cuda")
        ref = m.moe_layer_fwd(p, x, ws=ws)
        torch.cuda.synchronize()
        assert ws.status() == 0
        m.debug_stall_next_launch()
        t0 = time.perf_counter()
        m.moe_layer_fwd(p, x, ws=ws)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        assert ws.status() & m.STATUS_WAIT_TIMEOUT
        assert elapsed < 5.0
        again = m.moe_layer_fwd(p, x, ws=ws)
        torch.cuda.synchronize()
        assert ws.status() == 0
        diff = (again.double() - ref.double()).abs().max().item()
        assert diff <= 1e-2 * ref.double().abs().max().item()
    finally:
        m.set_wait_limit_ns(prev_limit)
        m.select_path(prev_path)


def test_stall_in_a_later_layer_then_recovers():
    """The stall at the start of layer 2 of a 3-layer stack: layers 0 and 1 ran
    (down-tile counters taken, activation buffers marked), then every CTA gave
    up. The status reports the timeout, and the next calls on the same
    workspace, a stack and a layer, give the results of a clean run."""
    import fine_grained_moe_gb300 as m
    prev_path = m.select_path(m.PATH_FUSED)
    prev_limit = m.set_wait_limit_ns(50_000_000)   # 50 ms
    try:
        ws = m.Workspace("cuda")
        layers = [synth.layer(l + 1, device="cuda", s=1.1) for l in range(3)]
        x = synth.hidden_states(6, 5, device="cuda")
        ref = m.moe_stack_fwd(layers, x, ws=ws)
        torch.cuda.synchronize()
        assert ws.status() == 0
        m.debug_stall_next_launch(2)
        m.moe_stack_fwd(layers, x, ws=ws)
        torch.cuda.synchronize()
        assert ws.status() & m.STATUS_WAIT_TIMEOUT
        # the grid barrier, or a producer waiting for the routing that the
        # barrier holds back: whichever checked the deadline first
        assert ws.wait_report()[0] in (6, 2)
        again = m.moe_stack_fwd(layers, x, ws=ws)
        torch.cuda.synchronize()
        assert ws.status() == 0
        diff = (again.double() - ref.double()).abs().max().item()
        assert diff <= 1e-2 * ref.double().abs().max().item()
        one = m.moe_layer_fwd(layers[0], x, ws=ws)
        torch.cuda.synchronize()
        assert ws.status() == 0
        assert torch.isfinite(one.float()).all()
    finally:
        m.set_wait_limit_ns(prev_limit)
        m.select_path(prev_path)
