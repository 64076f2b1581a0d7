"""The allocation-free layer call (fgm_moe_layer_fwd_noalloc).

It runs the same MoE layer as fgm_moe_layer_fwd on scratch built into the
library. The GPU test calls it twice in a row on different inputs and checks
each result against fgm_moe_layer_fwd with a caller workspace, under the same
rules as the oracle parity tests (rows within 1e-2 relative; router ids and
weights agree). The file is named to be collected last, so that it runs both
after the whole suite and, alone, in a fresh process.
"""

import gc
import ctypes

import numpy as np
import pytest
import torch

import synth
from helpers import REL_TOL, rowwise_rel_err


def _lib():
    """The library, built first when this file runs alone in a fresh tree."""
    import os

    import fine_grained_moe_gb300 as fgm
    if not os.path.exists(fgm.LIB_PATH):
        from fine_grained_moe_gb300 import build
        build.build()
    return fgm.lib()


def test_noalloc_rejects_m_beyond_its_scratch():
    import fine_grained_moe_gb300 as fgm
    L = fgm.fgm_layer()
    buf = (ctypes.c_uint8 * 4096)()
    lib = _lib()
    for M in (0, 9, 64):
        assert lib.fgm_moe_layer_fwd_noalloc(ctypes.byref(L), buf, buf, M, None, None, None) == -1
        assert b"at most 8 tokens" in lib.fgm_last_error()


@pytest.mark.gpu
def test_noalloc_matches_workspace_call_twice():
    import fine_grained_moe_gb300 as fgm
    prev = fgm.select_path(fgm.PATH_FUSED)
    try:
        p = synth.layer(0, device="cuda", s=1.1)
        ws = fgm.Workspace("cuda")
        cases = [(5, 7001), (8, 7002)]
        xs = [synth.hidden_states(seed, M, device="cuda") for M, seed in cases]
        ys = [torch.empty_like(x) for x in xs]
        ids = [torch.empty((x.shape[0], 8), dtype=torch.int32, device="cuda") for x in xs]
        wts = [torch.empty((x.shape[0], 8), dtype=torch.float32, device="cuda") for x in xs]
        # the first call on the device resolves the scratch address; the device
        # memory in use (torch's allocator and the driver's view of the whole
        # device) must not grow across the two calls that follow it
        fgm.moe_layer_fwd_noalloc(p, xs[0], ys[0])
        torch.cuda.synchronize()
        gc.collect()   # tensors of earlier tests freed now, not between the two readings
        before = torch.cuda.memory_allocated()
        free_before, _ = torch.cuda.mem_get_info()
        for i in range(2):   # two calls in a row on the built-in scratch
            fgm.moe_layer_fwd_noalloc(p, xs[i], ys[i], topk_ids=ids[i], topk_w=wts[i])
        torch.cuda.synchronize()
        free_after, _ = torch.cuda.mem_get_info()
        assert torch.cuda.memory_allocated() <= before
        assert free_after >= free_before
        for i, x in enumerate(xs):
            M = x.shape[0]
            rid = torch.empty((M, 8), dtype=torch.int32, device="cuda")
            rw = torch.empty((M, 8), dtype=torch.float32, device="cuda")
            ref = fgm.moe_layer_fwd(p, x, topk_ids=rid, topk_w=rw, ws=ws)
            torch.cuda.synchronize()
            ref64 = ref.float().cpu().numpy().astype(np.float64)
            assert rowwise_rel_err(ys[i], ref64).max() <= REL_TOL
            a, b = ids[i].cpu().numpy(), rid.cpu().numpy()
            for t in range(M):
                assert sorted(a[t].tolist()) == sorted(b[t].tolist())
            np.testing.assert_allclose(np.sort(wts[i].cpu().numpy(), axis=1),
                                       np.sort(rw.cpu().numpy(), axis=1), rtol=1e-5, atol=1e-7)
        assert ws.status() == 0
    finally:
        fgm.select_path(prev)
