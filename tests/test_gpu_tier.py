"""Routed experts in pinned host memory, gathered into HBM slots a token
ahead (HostTierStack): the same kernels on the same bytes, so every step's
output and routes equal the HBM-resident stack's bit for bit, eagerly and
through the captured graphs."""
import pytest
import torch

from int4_expert_gemv_gb300 import synth
from int4_expert_gemv_gb300.configs import ALL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    from int4_expert_gemv_gb300 import build
    build.build()
    from int4_expert_gemv_gb300 import moe
    moe.lib()
    synth._gpu()
    return moe


def test_host_tier_equals_hbm_stack(m):
    from int4_expert_gemv_gb300.model import DecodeStack, DeviceModel, HostTierStack
    cfg = ALL["35b-L4"]
    dm = DeviceModel(cfg)
    a, b = DecodeStack(dm), HostTierStack(dm)
    xs = [torch.from_numpy(synth.step_input(cfg, t)[0]).cuda() for t in range(8)]
    for t in range(8):
        if t == 3:
            a.capture()
            b.capture()
        a.step(xs[t])
        b.step(xs[t])
        torch.cuda.synchronize()
        assert torch.equal(a.stream, b.stream), t
        assert torch.equal(a.used_routes(t)[0], b.used_routes(t)[0]), t


def test_gather_marks_invalid_routes(m):
    """An index outside [0, E) is not copied and its slot index becomes n,
    which the expert call turns into NaN as it would the original index."""
    E, n, blob, stride = 8, 3, 4096, 4096
    pool = torch.arange(E * stride, dtype=torch.int64).to(torch.uint8).pin_memory()
    idx = torch.tensor([5, -1, 2], dtype=torch.int32, device="cuda")
    slots = torch.zeros(n * stride, dtype=torch.uint8, device="cuda")
    sidx = torch.full((n,), 99, dtype=torch.int32, device="cuda")
    m.moe_gather_experts(pool.data_ptr(), stride, E, idx, n, blob, slots, stride, sidx)
    torch.cuda.synchronize()
    assert sidx.tolist() == [0, n, 2]
    assert torch.equal(slots[:blob].cpu(), pool[5 * stride:5 * stride + blob])
    assert torch.equal(slots[2 * stride:2 * stride + blob].cpu(), pool[2 * stride:2 * stride + blob])
    assert int(slots[stride:2 * stride].sum()) == 0
