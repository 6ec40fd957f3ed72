"""Per-call parity of the CUDA path against the CPU oracle (needs a GPU).

Every call goes through the C ABI (libmoe.so via the ctypes binding); inputs
are seeded synthetic data from the generator module; expected values come
from the oracle only.  Bars: bit-exact decode and route indices, floating-point
outputs within max|err| <= 2e-3 * rms(ref).
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as orc
from int4_expert_gemv_gb300 import synth
from int4_expert_gemv_gb300.configs import ALL, MOE35B, TINY
from _util import TIE, assert_close, assert_close_bf16h, host_expert_from_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    from int4_expert_gemv_gb300 import build
    build.build()
    from int4_expert_gemv_gb300 import moe
    moe.lib()
    synth._gpu()
    return moe


def _f64(t):
    return t.detach().cpu().double().numpy()


# ------------------------------------------------------------ generator twin
@pytest.mark.parametrize("rows,cols,bits", [(64, 256, 4), (37, 128, 2), (5, 2048, 4), (3, 4096, 2)])
def test_generator_twin_is_bit_exact(m, rows, cols, bits):
    ref = synth.affine(7, 123, rows, cols, bits, 0.02)
    q = torch.empty((rows, cols * bits // 32), dtype=torch.int32, device="cuda")
    s = torch.empty((rows, cols // 64), dtype=torch.int16, device="cuda")
    b = torch.empty_like(s)
    synth.gpu_affine(7, 123, rows, cols, bits, 0.02, q, s, b)
    assert np.array_equal(q.cpu().numpy().view(np.uint32), ref["q"])
    assert np.array_equal(s.cpu().numpy().view(np.uint16), ref["s"])
    assert np.array_equal(b.cpu().numpy().view(np.uint16), ref["b"])
    g = synth.gpu_gauss(3, 9, torch.empty(10001, device="cuda"), 1.0)
    assert np.array_equal(g.cpu().numpy(), synth.gauss(3, 9, (10001,), 1.0))
    h = synth.gpu_gauss(3, 9, torch.empty(999, dtype=torch.int16, device="cuda"), 0.01)
    assert np.array_equal(h.cpu().numpy().view(np.uint16), synth.gauss_f16(3, 9, (999,), 0.01))


# ------------------------------------------------------------ decode
def _blob(m, cfg, e):
    ex = host_expert_from_gpu(cfg, 0, e)
    dev = lambda a: torch.from_numpy(a.view(np.int32) if a.dtype == np.uint32 else a.view(np.int16)).cuda()
    pool = torch.empty(m.moe_pool_expert_bytes(cfg.d, cfg.F, cfg.bits), dtype=torch.uint8, device="cuda")
    g, u, d = ex["gate"], ex["up"], ex["down"]
    m.moe_pack_experts(cfg.d, cfg.F, 1, cfg.bits, dev(g["q"]), dev(g["s"]), dev(g["b"]),
                       dev(u["q"]), dev(u["s"]), dev(u["b"]), dev(d["q"]), dev(d["s"]),
                       dev(d["b"]), pool, pool.numel())
    return ex, pool


@pytest.mark.parametrize("cfg", [TINY, MOE35B, ALL["wide-int2"]], ids=lambda c: c.name)
def test_packed_decode_is_bit_exact(m, cfg):
    ex, pool = _blob(m, cfg, 3)
    for which, key in enumerate(("gate", "up", "down")):
        mat = ex[key]
        out = torch.empty((mat["rows"], mat["cols"]), device="cuda")
        m.moe_debug_dequant(pool, cfg.d, cfg.F, cfg.bits, which, out)
        ref = orc.dequant(mat).astype(np.float32)   # exact in double, one rounding
        assert np.array_equal(out.cpu().numpy(), ref), key


# ------------------------------------------------------------ expert FFN
def _layer_model(cfg):
    from int4_expert_gemv_gb300.model import DeviceModel
    return DeviceModel(replace(cfg, L=1, depth=1), heads=False)


def _ffn_case(m, cfg, dm, routes, x_dtype=torch.float32, full=False):
    T, K = routes.shape
    ly = dm.layers[0]
    ed = ly["experts_desc"]
    x = torch.from_numpy(synth.gauss(cfg.seed, 777, (T, cfg.d), 1.0)).cuda().to(x_dtype)
    idx = torch.from_numpy(routes).cuda()
    y = torch.empty((T, K + cfg.shared, cfg.d), device="cuda")
    ws = torch.empty(m.moe_expert_ffn_workspace_bytes(ed, T, K), dtype=torch.uint8, device="cuda")
    m.moe_expert_ffn_int4(ed, x, idx, T, K, y, ws)
    needed = sorted(set(routes.ravel().tolist()))
    host = {e: host_expert_from_gpu(cfg, 0, e) for e in needed}
    zero = next(iter(host.values()))
    exps = [host.get(e, zero) for e in range(cfg.E)]
    sh = host_expert_from_gpu(cfg, 0, synth.SHARED_EXPERT) if cfg.shared else None
    xr = x.float().cpu().double().numpy()
    ref = orc.expert_ffn(exps, sh, xr, routes, round_h_bf16=x_dtype == torch.bfloat16)
    if full:
        return _f64(y), ref, exps, sh, xr
    return _f64(y), ref


@pytest.mark.parametrize("cfg", [TINY, MOE35B, ALL["8b"]], ids=lambda c: c.name)
def test_expert_ffn_decode_parity(m, cfg):
    dm = _layer_model(cfg)
    rng = np.random.default_rng(cfg.seed)
    for trial in range(3):
        routes = rng.permutation(cfg.E)[:cfg.K].astype(np.int32)[None]
        got, ref = _ffn_case(m, cfg, dm, routes)
        for s in range(ref.shape[1]):
            assert_close(got[0, s], ref[0, s], f"{cfg.name} trial {trial} slot {s}")


@pytest.mark.parametrize("bits", [4, 2])
def test_expert_ffn_wide_parity(m, bits):
    cfg = ALL[f"wide-int{bits}"]
    dm = _layer_model(cfg)
    routes = np.array([[511, 0, 200, 17]], np.int32)
    got, ref = _ffn_case(m, cfg, dm, routes)
    for s in range(cfg.K):
        assert_close(got[0, s], ref[0, s], f"wide int{bits} slot {s}")


def test_expert_ffn_repeated_expert_and_multi_token(m):
    cfg = TINY
    dm = _layer_model(cfg)
    routes = np.array([[3, 3], [15, 0], [7, 8], [0, 15], [1, 2]], np.int32)
    got, ref = _ffn_case(m, cfg, dm, routes)
    for t in range(routes.shape[0]):
        for s in range(cfg.K):
            assert_close(got[t, s], ref[t, s], f"token {t} slot {s}")
    assert np.array_equal(got[0, 0], got[0, 1])


def test_expert_ffn_bf16_activations(m):
    cfg = replace(MOE35B, T=8)
    dm = _layer_model(cfg)
    routes = synth.routes(4, 1, 8, cfg.E, cfg.K)
    got, ref, exps, sh, xr = _ffn_case(m, cfg, dm, routes, x_dtype=torch.bfloat16, full=True)
    for t in range(8):
        for s in range(cfg.slots):
            ex = exps[routes[t, s]] if s < cfg.K else sh
            assert_close_bf16h(got[t, s], ref[t, s], ex, xr[t], f"bf16 token {t} slot {s}")


# ------------------------------------------------------------ head
def _head_case(m, cfg, prec, T, with_prev=True, x_dtype=torch.float32):
    from int4_expert_gemv_gb300.model import DeviceModel
    c = replace(cfg, L=1, depth=1, head_prec=prec, E=cfg.E)
    dm = DeviceModel.__new__(DeviceModel)
    dm.cfg, dm.device = c, torch.device("cuda")
    hd = m.HeadDesc()
    hd.d, hd.E, hd.H = c.d, c.E, c.H
    hd.prec = m.MOE_PREC_FP16 if prec == "fp16" else m.MOE_PREC_AFFINE4
    tg = lambda k: synth.tag(k, 0)
    keep = dict(lx=DeviceModel._head_matrix(dm, synth.tag(synth.ROUTER, 0), c.E, c.d),
                fc1x=DeviceModel._head_matrix(dm, tg(synth.FC1X), c.H, c.d),
                fc2=DeviceModel._head_matrix(dm, tg(synth.FC2), c.E, c.H),
                fc1_tab=DeviceModel._f16(dm, tg(synth.FC1_TAB), (2 * c.E, c.H), c.sigma_w),
                b1=DeviceModel._f16(dm, tg(synth.B1), (c.H,), c.sigma_bias),
                b2=DeviceModel._f16(dm, tg(synth.B2), (c.E,), c.sigma_bias),
                l_tab=DeviceModel._f16(dm, tg(synth.L_TAB), (2 * c.E, c.E), c.sigma_w),
                bl=DeviceModel._f16(dm, tg(synth.BL), (c.E,), c.sigma_bias))
    for k, v in keep.items():
        setattr(hd, k, v.data_ptr())
    x = torch.from_numpy(synth.gauss(c.seed, 55, (T, c.d), 1.0)).cuda().to(x_dtype)
    cur = synth.routes(c.seed, 56, T, c.E, c.K)
    prev = synth.routes(c.seed, 57, T, c.E, c.K)
    logits = torch.empty((T, c.E), device="cuda")
    ws = torch.empty(m.moe_prerouter_head_workspace_bytes(hd, T), dtype=torch.uint8, device="cuda")
    m.moe_prerouter_head(hd, x, torch.from_numpy(cur).cuda(),
                         torch.from_numpy(prev).cuda() if with_prev else None, c.K, T, logits, ws)
    # oracle head from the host twin of the same tensors
    host = dict(d=c.d, E=c.E, H=c.H)
    hh = synth.head_host(replace(c, L=1), 0)
    host.update(hh)
    host["lx"] = synth.router_host(c, 0)["lx"]
    got = _f64(logits)
    for t in range(T):
        ref = orc.head_logits(host, x[t].float().cpu().double().numpy(), cur[t],
                              prev[t] if with_prev else None, c.K)
        assert_close(got[t], ref, f"head {c.name} {prec} token {t}")


@pytest.mark.parametrize("prec", ["int4", "fp16"])
@pytest.mark.parametrize("cfg", [TINY, MOE35B], ids=lambda c: c.name)
def test_prerouter_head_parity(m, cfg, prec):
    _head_case(m, cfg, prec, T=3)


@pytest.mark.parametrize("cfg,T", [(TINY, 100), (MOE35B, 64), (ALL["wide-int4"], 70)],
                         ids=["tiny-T100", "35b-T64", "wide-T70"])
@pytest.mark.parametrize("engine", [1, 2], ids=["mma_sync", "tcgen05"])
def test_prerouter_head_batched_bf16(m, cfg, T, engine):
    """Several bf16 tokens with an int4 head take the batched head (fc1 and l
    as one tensor-core job over all tokens), on either engine."""
    m.moe_debug_batched_engine(engine)
    try:
        _head_case(m, cfg, "int4", T, x_dtype=torch.bfloat16)
    finally:
        m.moe_debug_batched_engine(0)


def test_prerouter_head_without_prev_route(m):
    _head_case(m, TINY, "int4", T=2, with_prev=False)


def test_plain_router_parity(m):
    cfg = MOE35B
    r = synth.router_host(cfg, 0)
    from int4_expert_gemv_gb300.model import DeviceModel
    dm = DeviceModel.__new__(DeviceModel)
    dm.cfg, dm.device = cfg, torch.device("cuda")
    lx = DeviceModel._head_matrix(dm, synth.tag(synth.ROUTER, 0), cfg.E, cfg.d)
    hd = m.HeadDesc()
    hd.d, hd.E, hd.H, hd.prec, hd.lx = cfg.d, cfg.E, 0, m.MOE_PREC_AFFINE4, lx.data_ptr()
    x = torch.from_numpy(synth.gauss(1, 5, (2, cfg.d), 1.0)).cuda()
    logits = torch.empty((2, cfg.E), device="cuda")
    ws = torch.empty(max(256, m.moe_prerouter_head_workspace_bytes(hd, 2)), dtype=torch.uint8, device="cuda")
    m.moe_prerouter_head(hd, x, None, None, 4, 2, logits, ws)
    for t in range(2):
        assert_close(_f64(logits)[t], orc.head_logits(r, x[t].cpu().double().numpy()), "router")


# ------------------------------------------------------------ top-K
@pytest.mark.parametrize("E,K", [(16, 1), (16, 2), (256, 4), (256, 8), (512, 4), (1024, 16), (5, 5)])
def test_topk_route_parity(m, E, K):
    T = 64
    rng = np.random.default_rng(E * 100 + K)
    z = rng.normal(size=(T, E)).astype(np.float32)
    z[: T // 2] = np.round(z[: T // 2] * 2) / 2          # many exact ties
    zt = torch.from_numpy(z).cuda()
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), device="cuda")
    mg = torch.empty(T, device="cuda")
    m.moe_topk_route(zt, T, E, K, idx, w, mg)
    gi, gw, gm = idx.cpu().numpy(), _f64(w), _f64(mg)
    for t in range(T):
        ri, rw, rm = orc.topk(z[t].astype(np.float64), K)
        assert gi[t].tolist() == ri.tolist()                 # same fp32 inputs: exact
        assert np.allclose(gw[t], rw, rtol=1e-6, atol=1e-7)
        assert (rm == np.inf and gm[t] == np.inf) or abs(gm[t] - rm) <= 1e-6 * max(1.0, abs(rm))


# ------------------------------------------------------------ combine
@pytest.mark.parametrize("K,shared,xn", [(4, True, True), (2, False, True), (8, False, False), (1, True, False)])
def test_combine_parity(m, K, shared, xn):
    T, d = 3, 2048
    rng = np.random.default_rng(K)
    slots = K + shared
    y = rng.normal(size=(T, slots, d)).astype(np.float32)
    w = rng.dirichlet(np.ones(K), size=T).astype(np.float32)
    res = rng.normal(size=(T, d)).astype(np.float32)
    out = torch.empty((T, d), device="cuda")
    xnext = torch.empty((T, d), device="cuda") if xn else None
    m.moe_combine_residual(torch.from_numpy(y).cuda(), torch.from_numpy(w).cuda(), T, K, shared, d,
                           torch.from_numpy(res).cuda(), out, xnext)
    for t in range(T):
        ro, rx = orc.combine(y[t].astype(np.float64), w[t].astype(np.float64), shared,
                             res[t].astype(np.float64), want_x_next=True)
        assert_close(_f64(out)[t] - res[t], ro - res[t], "combine delta")
        if xn:
            assert_close(_f64(xnext)[t], rx, "x_next")


def test_combine_in_place_on_the_residual(m):
    T, K, d = 2, 4, 256
    rng = np.random.default_rng(0)
    y = torch.from_numpy(rng.normal(size=(T, K + 1, d)).astype(np.float32)).cuda()
    w = torch.full((T, K), 0.25, device="cuda")
    res = torch.from_numpy(rng.normal(size=(T, d)).astype(np.float32)).cuda()
    expect = res + (w[:, :, None] * y[:, :K]).sum(1) + y[:, K]
    m.moe_combine_residual(y, w, T, K, True, d, res, res)
    assert torch.allclose(res, expect, rtol=1e-5, atol=1e-5)


def test_empty_batch_writes_nothing(m):
    cfg = TINY
    dm = _layer_model(cfg)
    ed = dm.layers[0]["experts_desc"]
    y = torch.full((1, cfg.K, cfg.d), 7.0, device="cuda")
    ws = torch.empty(m.moe_expert_ffn_workspace_bytes(ed, 1, cfg.K), dtype=torch.uint8, device="cuda")
    m.moe_expert_ffn_int4(ed, torch.zeros((1, cfg.d), device="cuda"),
                          torch.zeros((1, cfg.K), dtype=torch.int32, device="cuda"), 0, cfg.K, y, ws)
    torch.cuda.synchronize()
    assert (y == 7.0).all()
