"""The allocation-free expert FFN entry point (moe_expert_ffn_int4_noalloc).

It serves callers that are handed only their input and output buffers and
cannot allocate device memory or carve out a workspace (a plugin inside a host
framework that owns the allocator, a real-time loop that forbids allocation
after start-up).  Its scratch is a fixed static device array inside the
library.  These tests call it through the C ABI and check that two calls in a
row agree with the regular entry point, which takes a caller workspace, within
the parity tolerance, and that its batched path (bf16 tokens sorted by
expert, grouped GEMMs over the static scratch) matches the oracle.  This file
sorts last so that a run stopping at the first failure has already run every
other test; it also passes on its own in a fresh process (it builds what it
needs).
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as orc
from int4_expert_gemv_gb300 import synth
from int4_expert_gemv_gb300.configs import MOE35B, TINY
from _util import assert_close, assert_close_bf16h, host_expert_from_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    from int4_expert_gemv_gb300 import build
    build.build()
    from int4_expert_gemv_gb300 import moe
    moe.lib()
    synth._gpu()
    return moe


@pytest.mark.parametrize("cfg,T", [(TINY, 1), (MOE35B, 1), (MOE35B, 8)], ids=["tiny", "35b", "35b-T8"])
def test_noalloc_matches_workspace_entry_point_twice(m, cfg, T):
    from int4_expert_gemv_gb300.model import DeviceModel
    c = replace(cfg, L=1, depth=1)
    dm = DeviceModel(c, heads=False)
    ed = dm.layers[0]["experts_desc"]
    ws = torch.empty(m.moe_expert_ffn_workspace_bytes(ed, T, c.K), dtype=torch.uint8, device="cuda")
    assert m.moe_expert_ffn_workspace_bytes(ed, T, c.K) <= m.MOE_FFN_STATIC_SCRATCH_BYTES
    for call in range(2):                      # two calls in a row, different inputs
        x = torch.from_numpy(synth.gauss(c.seed, 900 + call, (T, c.d), 1.0)).cuda()
        idx = torch.from_numpy(synth.routes(c.seed, 950 + call, T, c.E, c.K)).cuda()
        y_ref = torch.empty((T, c.slots, c.d), device="cuda")
        y_new = torch.full((T, c.slots, c.d), float("nan"), device="cuda")
        m.moe_expert_ffn_int4(ed, x, idx, T, c.K, y_ref, ws)
        m.moe_expert_ffn_int4_noalloc(ed, x, idx, T, c.K, y_new)
        torch.cuda.synchronize()
        got, ref = y_new.cpu().double().numpy(), y_ref.cpu().double().numpy()
        for t in range(T):
            for s in range(c.slots):
                assert_close(got[t, s], ref[t, s], f"noalloc call {call} token {t} slot {s}")


@pytest.mark.parametrize("T", [8, 64])
def test_noalloc_batched_bf16_matches_the_oracle_twice(m, T):
    """bf16 tokens take the batched path (sort by expert, grouped GEMMs),
    whose sort buffers, gathered x, h and status word all live in the static
    scratch: two calls in a row against the oracle, and the status word
    read back through moe_expert_ffn_noalloc_status."""
    from int4_expert_gemv_gb300.model import DeviceModel
    c = replace(MOE35B, L=1, depth=1, seed=4)
    dm = DeviceModel(c, heads=False)
    ed = dm.layers[0]["experts_desc"]
    assert m.moe_expert_ffn_workspace_bytes(ed, T, c.K) <= m.MOE_FFN_STATIC_SCRATCH_BYTES
    for call in range(2):
        x = torch.from_numpy(synth.gauss(c.seed, 960 + call, (T, c.d), 1.0)).cuda().to(torch.bfloat16)
        routes = synth.routes(c.seed, 970 + call, T, c.E, c.K)
        y = torch.full((T, c.slots, c.d), float("nan"), device="cuda")
        m.moe_expert_ffn_int4_noalloc(ed, x, torch.from_numpy(routes).cuda(), T, c.K, y)
        assert m.moe_expert_ffn_noalloc_status() == m.MOE_OK
        got = y.cpu().double().numpy()
        tokens = np.arange(0, T, max(1, T // 8))
        need = sorted(set(routes[tokens].ravel().tolist()))
        host = {e: host_expert_from_gpu(c, 0, e) for e in need}
        exps = [host.get(e, host[need[0]]) for e in range(c.E)]
        sh = host_expert_from_gpu(c, 0, synth.SHARED_EXPERT)
        xr = x.float().cpu().double().numpy()[tokens]
        ref = orc.expert_ffn(exps, sh, xr, routes[tokens], round_h_bf16=True)
        for i, t in enumerate(tokens):
            for s_ in range(c.slots):
                ex = exps[routes[t, s_]] if s_ < c.K else sh
                assert_close_bf16h(got[t, s_], ref[i, s_], ex, xr[i],
                                   f"noalloc batched call {call} token {t} slot {s_}")


def test_noalloc_rejects_batches_beyond_the_static_scratch(m):
    from int4_expert_gemv_gb300.model import DeviceModel
    c = replace(MOE35B, L=1, depth=1)
    dm = DeviceModel(c, heads=False)
    ed = dm.layers[0]["experts_desc"]
    T = 4096
    assert m.moe_expert_ffn_workspace_bytes(ed, T, c.K) > m.MOE_FFN_STATIC_SCRATCH_BYTES
    x = torch.zeros((T, c.d), device="cuda")
    idx = torch.zeros((T, c.K), dtype=torch.int32, device="cuda")
    y = torch.empty((T, c.slots, c.d), device="cuda")
    with pytest.raises(m.MoEError) as e:
        m.moe_expert_ffn_int4_noalloc(ed, x, idx, T, c.K, y)
    assert e.value.status == m.MOE_ENOSPACE
    assert "static scratch" in str(e.value)
