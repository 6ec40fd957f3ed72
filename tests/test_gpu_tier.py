"""Routed experts in pinned host memory, brought into HBM a token ahead.

HostTierStack (per-call path, slots per step) and HostTierChain (chained
step, an LRU cache of experts per layer): the chained tier is compared with
the oracle's stack step, and both with the HBM-resident stacks bit for bit
(the same kernels on the same bytes), eagerly and through captured graphs;
the cache's decisions are checked against a plain model of its rule."""
import numpy as np
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


@pytest.mark.parametrize("slots,free_sms", [(5, 0), (16, 24)])
def test_host_tier_chain_matches_the_oracle(m, slots, free_sms):
    """The chained step reading its experts from per-layer HBM caches of a
    few slots (many misses and evictions; slots >= K + 1 so a route never
    evicts itself) against the oracle's stack step, 6 steps; also with SMs
    left free for the copies (the step's kernels then split the work over
    fewer CTAs)."""
    from test_gpu_stack import check_stack
    from int4_expert_gemv_gb300.model import HostTierChain
    check_stack(ALL["35b-L4"], 6, make=lambda dm: HostTierChain(dm, slots, free_sms))


def test_host_tier_chain_equals_hbm_chain(m):
    from int4_expert_gemv_gb300.model import DecodeStack, DeviceModel, HostTierChain
    cfg = ALL["35b-L4"]
    dm = DeviceModel(cfg)
    a, b = DecodeStack(dm, fused="chain"), HostTierChain(dm, 12)
    xs = [torch.from_numpy(synth.step_input(cfg, t)[0]).cuda() for t in range(10)]
    for t in range(10):
        if t == 4:
            a.capture()
            b.capture()
        a.step(xs[t])
        b.step(xs[t])
        torch.cuda.synchronize()
        assert torch.equal(a.stream, b.stream), t
        assert torch.equal(a.used_routes(t)[0], b.used_routes(t)[0]), t
    assert b.status() == m.MOE_OK
    hits, misses = b.stats.sum(0).tolist()
    assert misses > 0 and hits + misses <= (cfg.depth - 1) * cfg.K * 10


def _lru_model(routes, E, C):
    """The cache rule written out on the host: per route, hits keep their
    slot; each other valid expert takes the unpinned slot with the smallest
    (occupied, age, index); the route's slots get the call's step."""
    tags, ages = [-1] * C, [0] * C
    out = []
    for step, route in enumerate(routes, 1):
        pinned, slots, hits, misses, copies = set(), [], 0, 0, []
        for i, e in enumerate(route):
            if not 0 <= e < E:
                slots.append(C)
                continue
            if e in tags:
                s = tags.index(e)
                if e not in route[:i]:
                    hits += 1
            else:
                s = min((j for j in range(C) if j not in pinned),
                        key=lambda j: (tags[j] >= 0, ages[j], j))
                tags[s] = e
                misses += 1
                copies.append((e, s))
            pinned.add(s)
            ages[s] = step
            slots.append(s)
        out.append((slots, hits, misses, copies))
    return out


def test_cache_decisions_follow_the_lru_rule(m):
    E, C, n, blob, stride = 16, 6, 3, 4096, 4096
    pool = torch.arange(E * stride, dtype=torch.int64).to(torch.uint8).pin_memory()
    rng = np.random.default_rng(5)
    routes = [rng.choice(E, n, replace=False).tolist() for _ in range(12)]
    routes[4] = [7, 7, 2]                       # a repeated expert
    routes[6] = [3, -1, E + 2]                  # indices outside [0, E)
    i32 = dict(dtype=torch.int32, device="cuda")
    cache = torch.zeros(C * stride, dtype=torch.uint8, device="cuda")
    tags, ages, clock = torch.full((C,), -1, **i32), torch.zeros(C, **i32), torch.zeros(1, **i32)
    sidx, plan, stats = torch.zeros(n, **i32), torch.zeros(n, **i32), torch.zeros(2, **i32)
    want = _lru_model(routes, E, C)
    for route, (slots, hits, misses, copies) in zip(routes, want):
        before = stats.clone()
        m.moe_cache_experts(pool.data_ptr(), stride, E, torch.tensor(route, **i32), n, blob, cache,
                            stride, C, tags, ages, clock, sidx, plan, stats)
        torch.cuda.synchronize()
        assert sidx.tolist() == slots, route
        assert (stats - before).tolist() == [hits, misses], route
        for e, s in copies:
            assert torch.equal(cache[s * stride:s * stride + blob].cpu(), pool[e * stride:e * stride + blob])
    assert clock.item() == len(routes)
