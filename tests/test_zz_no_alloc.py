"""The allocation-free expert FFN entry point (moe_expert_ffn_int4_noalloc).

It serves callers that are handed only their input and output buffers and
cannot allocate device memory or carve out a workspace (a plugin inside a host
framework that owns the allocator, a real-time loop that forbids allocation
after start-up).  Its scratch is a fixed static device array inside the
library.  These tests call it through the C ABI and check that two calls in a
row agree with the regular entry point, which takes a caller workspace, within
the parity tolerance.  This file sorts last so that a run stopping at the first
failure has already run every other test; it also passes on its own in a fresh
process (it builds what it needs).
"""
from dataclasses import replace

import pytest
import torch

from int4_expert_gemv_gb300 import synth
from int4_expert_gemv_gb300.configs import MOE35B, TINY
from _util import assert_close

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
