"""Batched / prefill expert FFN (T > 1 tokens, bf16 activations): the grouped
path (counting sort by expert, grouped tensor-core GEMMs) against the oracle.

Calls go through the C ABI; routes come from the seeded generator; expected
values from the oracle only, with h rounded to bf16 on both sides (where
the oracle's h sits within 1e-5 of a rounding midpoint either neighbour is
accepted, and the bar widens by what that choice can move).  Up to
T = 64 every token is compared; at T = 512 and 4096 a seeded sample of tokens
(all their slots) is, since each (token, slot) output depends only on that
token's row of x and its expert.  Bar: max|err| <= 2e-3 * rms(ref) per slot."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as orc
from int4_expert_gemv_gb300 import synth
from int4_expert_gemv_gb300.configs import ALL, TINY
from _util import (TIE, TOL, assert_close, assert_close_bf16h, bf16_h_allowance,
                   host_expert_from_gpu, rms)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    from int4_expert_gemv_gb300 import build
    build.build()
    from int4_expert_gemv_gb300 import moe
    moe.lib()
    synth._gpu()
    return moe


_MODELS = {}


@pytest.fixture(params=[1, 2], ids=["mma_sync", "tcgen05"])
def engine(request, m):
    """Both engines of the grouped GEMMs: the register engine (mma.sync) and
    the tensor-memory engine (tcgen05.mma, TMEM accumulators)."""
    m.moe_debug_batched_engine(request.param)
    yield request.param
    m.moe_debug_batched_engine(0)


def _model(cfg):
    from int4_expert_gemv_gb300.model import DeviceModel
    key = (cfg.d, cfg.F, cfg.E, cfg.bits, cfg.shared, cfg.seed, cfg.lora_on, cfg.lora_r)
    if key not in _MODELS:
        _MODELS.clear()
        torch.cuda.empty_cache()
        _MODELS[key] = DeviceModel(replace(cfg, L=1, depth=1), heads=False)
    return _MODELS[key]


def _run(m, cfg, routes, x):
    T, K = routes.shape
    ed = _model(cfg).layers[0]["experts_desc"]
    y = torch.full((T, K + cfg.shared, cfg.d), 7.0, device="cuda")
    ws = torch.empty(m.moe_expert_ffn_workspace_bytes(ed, T, K), dtype=torch.uint8, device="cuda")
    m.moe_expert_ffn_int4(ed, x, torch.from_numpy(routes).cuda(), T, K, y, ws)
    torch.cuda.synchronize()
    if T > 1:      # the batched path's status word (the decode path has none)
        assert ws[:4].view(torch.int32).item() == m.MOE_OK     # no bounded wait expired
    return y.cpu().double().numpy()


def _x(cfg, T, tag=901):
    return torch.from_numpy(synth.gauss(cfg.seed, tag, (T, cfg.d), 1.0)).cuda().to(torch.bfloat16)


def _check(cfg, got, x, routes, tokens, what):
    valid = (routes >= 0) & (routes < cfg.E)
    safe = np.where(valid, routes, 0).astype(np.int32)
    needed = sorted(set(safe[tokens].ravel().tolist()))
    host = {e: host_expert_from_gpu(cfg, 0, e) for e in needed}
    zero = next(iter(host.values()))
    exps = [host.get(e, zero) for e in range(cfg.E)]
    sh = host_expert_from_gpu(cfg, 0, synth.SHARED_EXPERT) if cfg.shared else None
    xr = x.float().cpu().double().numpy()[tokens]
    ref = orc.expert_ffn(exps, sh, xr, safe[tokens], round_h_bf16=True)
    for i, t in enumerate(tokens):
        for s in range(ref.shape[1]):
            if s < cfg.K and not valid[t, s]:
                assert np.isnan(got[t, s]).all(), f"{what}: token {t} slot {s} not NaN"
                continue
            ex = exps[safe[t, s]] if s < cfg.K else sh
            assert_close_bf16h(got[t, s], ref[i, s], ex, xr[i], f"{what} token {t} slot {s}")


@pytest.mark.parametrize("T,sample", [(8, 0), (64, 0), (512, 48), (4096, 24)])
def test_batched_parity(m, engine, T, sample):
    cfg = ALL[f"batched-T{T}"]
    routes = synth.routes(cfg.seed, 902, T, cfg.E, cfg.K)
    x = _x(cfg, T)
    got = _run(m, cfg, routes, x)
    assert np.isfinite(got).all()
    tokens = np.arange(T) if not sample else np.sort(
        np.random.default_rng(T).choice(T, sample, replace=False))
    _check(cfg, got, x, routes, tokens, f"batched T={T}")


def test_batched_is_deterministic(m):
    cfg = ALL["batched-T512"]
    routes = synth.routes(cfg.seed, 903, 512, cfg.E, cfg.K)
    x = _x(cfg, 512)
    a = _run(m, cfg, routes, x)
    b = _run(m, cfg, routes, x)
    assert np.array_equal(a.view(np.int64), b.view(np.int64))


def test_batched_ragged_tiny_with_invalid_and_repeated(m, engine):
    """T not a multiple of the 64-token tile, F below the 256-column chunk,
    LoRA on the routed down projection, expert indices outside [0, E) (NaN
    slots) and an expert repeated within a token."""
    cfg = TINY
    T = 100
    routes = synth.routes(cfg.seed, 904, T, cfg.E, cfg.K)
    routes[3] = [5, 5]
    routes[10, 1] = -1
    routes[57, 0] = cfg.E
    routes[99] = [cfg.E + 7, 2]
    x = _x(cfg, T)
    got = _run(m, cfg, routes, x)
    _check(cfg, got, x, routes, np.arange(T), "tiny ragged")
    assert np.array_equal(got[3, 0], got[3, 1])


def test_batched_one_expert_beyond_the_tile_grid(m, engine):
    """Every slot of every token on one expert: the expert has T*K entries,
    more than the grid's ceil(T/64) tiles cover in one pass."""
    cfg = TINY
    T = 70
    routes = np.full((T, cfg.K), 9, np.int32)
    x = _x(cfg, T, 905)
    got = _run(m, cfg, routes, x)
    _check(cfg, got, x, routes, np.arange(0, T, 3), "one expert")
    assert np.array_equal(got[:, 0], got[:, 1])


@pytest.mark.parametrize("bits", [2, 4])
def test_batched_wide(m, engine, bits):
    cfg = replace(ALL[f"wide-int{bits}"], T=64)
    routes = synth.routes(cfg.seed, 906, 64, cfg.E, cfg.K)
    for t in range(8):                   # one expert with 8 tokens, indices still distinct
        row = [77] + [e for e in routes[t] if e != 77]
        routes[t] = row[:cfg.K]
    x = _x(cfg, 64)
    got = _run(m, cfg, routes, x)
    _check(cfg, got, x, routes, np.arange(0, 64, 4), f"wide int{bits}")


def test_batched_matches_per_token_bf16_path(m):
    """The grouped path and the per-token GEMV path (one call per token) take
    the same arithmetic definition: both agree within the bar."""
    cfg = ALL["batched-T64"]
    routes = synth.routes(cfg.seed, 907, 64, cfg.E, cfg.K)
    x = _x(cfg, 64)
    got = _run(m, cfg, routes, x)
    sh = host_expert_from_gpu(cfg, 0, synth.SHARED_EXPERT)
    for t in (0, 17, 63):
        one = _run(m, cfg, routes[t:t + 1], x[t:t + 1].contiguous())
        xr = x[t].float().cpu().double().numpy()
        for s in range(cfg.slots):
            ex = host_expert_from_gpu(cfg, 0, int(routes[t, s])) if s < cfg.K else sh
            assert_close_bf16h(got[t, s], one[0, s], ex, xr,
                               f"grouped vs per-token token {t} slot {s}")


def test_batched_layer_step(m):
    """The whole batched layer (head + top-K over T rows, grouped expert FFN,
    combine + residual) against the oracle, on sampled tokens: next-layer
    routes as index sets where the oracle's margin exceeds the tie bar, their
    weights, and the layer output (minus the residual)."""
    from int4_expert_gemv_gb300.model import BatchedLayer, DeviceModel
    _MODELS.clear()
    cfg = ALL["batched-T64"]
    T = cfg.T
    bl = BatchedLayer(DeviceModel(cfg), T)
    x0 = torch.from_numpy(synth.gauss(cfg.seed, 908, (T, cfg.d), 1.0)).cuda()
    bl.x.copy_(x0.to(torch.bfloat16))
    bl.res.copy_(x0)
    bl.route_own()
    bl.enqueue()
    torch.cuda.synchronize()
    cur, cw, prev = (a.cpu().numpy() for a in (bl.cur_idx, bl.cur_w, bl.prev_idx))
    nidx, nw = bl.next_idx.cpu().numpy(), bl.next_w.cpu().double().numpy()
    out = bl.out.cpu().double().numpy()
    xb = bl.x.float().cpu().double().numpy()
    res = x0.cpu().double().numpy()
    head = synth.head_host(cfg, 0)
    sh = host_expert_from_gpu(cfg, 0, synth.SHARED_EXPERT)
    checked = 0
    for t in range(0, T, 7):
        z = orc.head_logits(head, xb[t], cur[t], prev[t], cfg.K)
        idx, w, margin = orc.topk(z, cfg.K)
        if margin > TIE:
            checked += 1
            assert set(idx.tolist()) == set(nidx[t].tolist()), t
            gw = dict(zip(nidx[t].tolist(), nw[t]))
            assert_close([gw[k] for k in idx.tolist()], w, f"next weights token {t}")
        exps = {e: host_expert_from_gpu(cfg, 0, int(e)) for e in cur[t]}
        lst = [exps.get(e, sh) for e in range(cfg.E)]
        y = orc.expert_ffn(lst, sh, xb[t:t + 1], cur[t:t + 1], round_h_bf16=True)[0]
        ref, _ = orc.combine(y, cw[t].astype(np.float64), True, res[t])
        got_d, ref_d = out[t] - res[t], ref - res[t]
        err = np.abs(got_d - ref_d)
        bound = TOL * rms(ref_d)
        if err.max() > bound:
            allow = sum(float(cw[t, k]) * bf16_h_allowance(exps[cur[t, k]], xb[t])
                        for k in range(cfg.K)) + bf16_h_allowance(sh, xb[t])
            assert (err <= bound + allow).all(), f"layer output token {t}"
    assert checked >= 6


def test_batched_bounded_wait_times_out_and_recovers(m):
    """The batched engine's waits take the set limit: with the test hook on,
    one consumer warp waits for bytes no copy sends; after 50 ms MOE_ETIMEOUT
    lands in ws word 0 and the launches return (the context stays usable).
    With the hook off the next call's outputs match the oracle again."""
    import time
    cfg = ALL["batched-T64"]
    T = 64
    routes = synth.routes(cfg.seed, 907, T, cfg.E, cfg.K)
    x = _x(cfg, T, 908)
    ed = _model(cfg).layers[0]["experts_desc"]
    y = torch.full((T, cfg.slots, cfg.d), 7.0, device="cuda")
    ws = torch.empty(m.moe_expert_ffn_workspace_bytes(ed, T, cfg.K), dtype=torch.uint8, device="cuda")
    m.moe_debug_batched_waits(50_000_000, True)
    try:
        t0 = time.time()
        m.moe_expert_ffn_int4(ed, x, torch.from_numpy(routes).cuda(), T, cfg.K, y, ws)
        torch.cuda.synchronize()                                    # context alive
        assert ws[:4].view(torch.int32).item() == m.MOE_ETIMEOUT
        assert time.time() - t0 < 10.0               # the 50 ms limit, not 1 s per wait
    finally:
        m.moe_debug_batched_waits(0, False)
    got = _run(m, cfg, routes, x)                    # asserts MOE_OK in ws word 0
    _check(cfg, got, x, routes, np.arange(0, T, 4), "batched after a timed-out call")
