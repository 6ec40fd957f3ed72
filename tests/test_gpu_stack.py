"""Decode-stack parity: the CUDA path (four C-ABI calls per layer, steady-state
steps replayed from captured CUDA graphs, exactly as bench.py times them)
against the oracle's stack step, on the full-size configurations.

Routes: compared as index sets per layer wherever the oracle's K-th/(K+1)-th
logit margin exceeds 1e-4; at nearer ties the oracle adopts the GPU's route
(teacher forcing) and recomputes its own weights there.  Weights are compared
per index, outputs as the MoE delta (final stream minus the step input)."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as orc
from int4_expert_gemv_gb300 import synth
from int4_expert_gemv_gb300.configs import ALL, TINY
from _util import TIE, assert_close, host_expert_from_gpu, zero_expert

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from int4_expert_gemv_gb300 import build
    build.build()


def run_gpu(cfg, steps, fused=False, make=None):
    """Run `steps` decode steps (captured graphs from step 1 on) and record
    each step's routes and output.  make(model): another stack driver to run
    (default: DecodeStack on the path `fused` names)."""
    from int4_expert_gemv_gb300 import moe
    from int4_expert_gemv_gb300.model import DecodeStack, DeviceModel
    dm = DeviceModel(cfg)
    cluster = fused == "cluster"
    if cluster:
        moe.moe_decode_step_chain_variant(2)
        fused = "chain"
    try:
        st = make(dm) if make is not None else DecodeStack(dm, fused=fused)
        rec = []
        for t in range(steps):
            x0 = torch.from_numpy(synth.step_input(cfg, t)[0]).cuda()
            st.step(x0)
            if t == 0:
                st.capture()
            idx, w, mg = st.used_routes(t)
            torch.cuda.synchronize()
            rec.append(dict(idx=idx.cpu().numpy(), w=w.cpu().double().numpy(),
                            margin=mg.cpu().double().numpy(), out=st.stream.cpu().double().numpy()))
        if st.fused:
            assert st.status() == 0
    finally:
        if cluster:
            moe.moe_decode_step_chain_variant(0)
    del st, dm
    torch.cuda.empty_cache()
    return rec


def oracle_layers(cfg, rec):
    used = {r: set() for r in range(cfg.L)}
    for r_ in rec:
        for N in range(cfg.depth):
            used[N % cfg.L].update(r_["idx"][N].tolist())
    zero = zero_expert(cfg)
    res = []
    for r in range(cfg.L):
        exps = {e: host_expert_from_gpu(cfg, r, e) for e in sorted(used[r])}
        res.append(dict(experts=[exps.get(e, zero) for e in range(cfg.E)],
                        shared=host_expert_from_gpu(cfg, r, synth.SHARED_EXPERT) if cfg.shared else None,
                        router=synth.router_host(cfg, r), head=synth.head_host(cfg, r)))
    return [res[N % cfg.L] for N in range(cfg.depth)]


def check_stack(cfg, steps, fused=False, make=None):
    rec = run_gpu(cfg, steps, fused, make)
    run = orc.StackRunner(oracle_layers(cfg, rec), cfg.d, cfg.E, cfg.K,
                          single_layer_self_predict=cfg.self_predict)
    forced = 0
    for t, g in enumerate(rec):
        x0 = synth.step_input(cfg, t)[0].astype(np.float64)
        r = run.step(x0, ext_idx=g["idx"], tie_margin=TIE)
        for N in range(cfg.depth):
            if r["forced"][N]:
                forced += 1
                assert r["margin"][N] <= TIE
                continue
            assert set(g["idx"][N].tolist()) == set(r["idx"][N].tolist()), (t, N)
            gw = dict(zip(g["idx"][N].tolist(), g["w"][N]))
            rw = dict(zip(r["idx"][N].tolist(), r["w"][N]))
            keys = sorted(rw)
            assert_close([gw[k] for k in keys], [rw[k] for k in keys], f"weights t{t} N{N}")
        assert_close(g["out"] - x0, r["out"] - x0, f"{cfg.name} step {t} output delta")
    return forced


PATHS = [pytest.param(False, id="per-call"), pytest.param(True, id="fused"),
         pytest.param("chain", id="chain"), pytest.param("cluster", id="cluster")]


@pytest.mark.parametrize("fused", PATHS)
def test_tiny_stack_all_steps(fused):
    forced = check_stack(TINY, TINY.steps, fused)
    assert forced <= TINY.steps // 8           # near-ties are rare


@pytest.mark.parametrize("fused", PATHS)
def test_35b_stack_full_size(fused):
    check_stack(ALL["35b"], 4, fused)


@pytest.mark.parametrize("fused", PATHS)
def test_8b_stack_full_size(fused):
    check_stack(ALL["8b"], 2, fused)


@pytest.mark.parametrize("fused", PATHS)
@pytest.mark.parametrize("name", ["wide-int4", "wide-int2"])
def test_wide_stack_full_size(name, fused):
    if fused == "cluster":
        pytest.skip("a CTA's share of a wide slot does not fit shared memory (two-kernel chain)")
    check_stack(ALL[name], 2, fused)


@pytest.mark.parametrize("fused", PATHS)
def test_k_sweep_stack(fused):
    for K in (2, 8):
        check_stack(replace(ALL[f"35b-K{K}"], L=4, depth=4), 3, fused)


def test_fused_bounded_wait_times_out_and_recovers():
    """A wait on a flag nothing sets runs out after its short limit; the kernel
    records MOE_ETIMEOUT and returns, the context stays usable, and a zeroed
    workspace runs the next step normally."""
    from int4_expert_gemv_gb300 import moe
    from int4_expert_gemv_gb300.model import DecodeStack, DeviceModel
    cfg = TINY
    st = DecodeStack(DeviceModel(cfg), fused=True)
    st.step(torch.from_numpy(synth.step_input(cfg, 0)[0]).cuda())       # step 0: per-call
    st.sd.timeout_ns = 50_000_000
    st.sd.debug_unset_wait = 1
    st.step(torch.from_numpy(synth.step_input(cfg, 1)[0]).cuda())
    assert st.status() == moe.MOE_ETIMEOUT
    torch.cuda.synchronize()                                               # context alive
    st.sd.debug_unset_wait = 0
    st.sd.timeout_ns = 0
    st.step_ws.zero_()
    st.t = 1
    st.step(torch.from_numpy(synth.step_input(cfg, 1)[0]).cuda())
    assert st.status() == moe.MOE_OK
    assert torch.isfinite(st.stream).all()


def test_chain_bounded_wait_times_out_and_recovers():
    """The chained step's mbarrier waits take the caller's limit: with the
    test hook on, CTA 0 of layer 0's first kernel waits for bytes no copy
    sends; after the 50 ms limit MOE_ETIMEOUT lands in the status word and
    the kernel returns (the context stays usable).  Step 1 run again with the
    hook off, then steps 2 and 3, give the same bits as a stack that never
    stalled (whose path the stack tests compare with the oracle)."""
    import time
    from int4_expert_gemv_gb300 import moe
    from int4_expert_gemv_gb300.model import DecodeStack, DeviceModel
    cfg = ALL["35b-L4"]
    dm = DeviceModel(cfg)
    st, ref = DecodeStack(dm, fused="chain"), DecodeStack(dm, fused="chain")
    xs = [torch.from_numpy(synth.step_input(cfg, t)[0]).cuda() for t in range(4)]
    st.step(xs[0])                                                         # step 0: per-call
    ref.step(xs[0])
    st.sd.timeout_ns = 50_000_000
    st.sd.debug_unset_wait = 1
    t0 = time.time()
    st.step(xs[1])
    assert st.status() == moe.MOE_ETIMEOUT
    assert time.time() - t0 < 10.0                   # the 50 ms limit, not 1 s per wait
    torch.cuda.synchronize()                                               # context alive
    st.sd.debug_unset_wait = 0
    st.sd.timeout_ns = 0
    st.t = 1
    for t in (1, 2, 3):
        st.step(xs[t])
        ref.step(xs[t])
        assert st.status() == moe.MOE_OK
        assert torch.equal(st.stream, ref.stream)
        assert torch.equal(st.r_idx, ref.r_idx)
    assert torch.isfinite(st.stream).all()


def test_cluster_bounded_wait_times_out_and_recovers():
    """The cluster form of the chained step: with the test hook on, CTA 0 of
    layer 0 waits for bytes no copy sends; after the 50 ms limit MOE_ETIMEOUT
    lands in the status word.  The CTA then carries on (its cluster peers'
    waits for its h run out the same way), every CTA reaches the cluster
    barrier and the step ends; steps run again with the hook off give the
    same bits as a stack that never stalled."""
    import time
    from int4_expert_gemv_gb300 import moe
    from int4_expert_gemv_gb300.model import DecodeStack, DeviceModel
    cfg = ALL["35b-L4"]
    dm = DeviceModel(cfg)
    moe.moe_decode_step_chain_variant(2)
    try:
        st, ref = DecodeStack(dm, fused="chain"), DecodeStack(dm, fused="chain")
        xs = [torch.from_numpy(synth.step_input(cfg, t)[0]).cuda() for t in range(4)]
        st.step(xs[0])                                                     # step 0: per-call
        ref.step(xs[0])
        st.sd.timeout_ns = 50_000_000
        st.sd.debug_unset_wait = 1
        t0 = time.time()
        st.step(xs[1])
        assert st.status() == moe.MOE_ETIMEOUT
        assert time.time() - t0 < 10.0
        torch.cuda.synchronize()                                           # context alive
        st.sd.debug_unset_wait = 0
        st.sd.timeout_ns = 0
        st.t = 1
        for t in (1, 2, 3):
            st.step(xs[t])
            ref.step(xs[t])
            assert st.status() == moe.MOE_OK
            assert torch.equal(st.stream, ref.stream)
            assert torch.equal(st.r_idx, ref.r_idx)
    finally:
        moe.moe_decode_step_chain_variant(0)


def test_chain_graph_cache_gives_the_same_bits():
    """moe_decode_step_chain replays repeated calls from its graph cache (on
    by default): the routes and outputs of 8 steps (every t mod 3, several
    hits per key) equal, bit for bit, those of the same calls run directly
    (cache off), on both forms of the step."""
    from int4_expert_gemv_gb300 import moe
    from int4_expert_gemv_gb300.model import DecodeStack, DeviceModel
    cfg = ALL["35b-L4"]
    dm = DeviceModel(cfg)
    xs = [torch.from_numpy(synth.step_input(cfg, t)[0]).cuda() for t in range(8)]
    try:
        for variant in (1, 2):
            moe.moe_decode_step_chain_variant(variant)
            res = {}
            for cache in (16, 0):
                moe.moe_decode_step_chain_cache(cache)
                st = DecodeStack(dm, fused="chain")
                res[cache] = []
                for t in range(8):
                    st.step(xs[t])
                    res[cache].append((st.stream.clone(), st.r_idx.clone(), st.r_w.clone()))
                assert st.status() == moe.MOE_OK
            for a, b in zip(res[16], res[0]):
                for u, v in zip(a, b):
                    assert torch.equal(u, v)
    finally:
        moe.moe_decode_step_chain_variant(0)
        moe.moe_decode_step_chain_cache(16)


def test_cluster_variant_rejects_what_does_not_fit():
    """The wide shapes' slot shares do not fit a CTA: the cluster form
    reports MOE_EUNSUPPORTED before enqueueing anything."""
    from int4_expert_gemv_gb300 import moe
    from int4_expert_gemv_gb300.model import DecodeStack, DeviceModel
    cfg = replace(ALL["wide-int4"], L=1, depth=2)
    st = DecodeStack(DeviceModel(cfg), fused="chain")
    st.step(torch.from_numpy(synth.step_input(cfg, 0)[0]).cuda())
    moe.moe_decode_step_chain_variant(2)
    try:
        with pytest.raises(RuntimeError, match="MOE_EUNSUPPORTED"):
            st.step(torch.from_numpy(synth.step_input(cfg, 1)[0]).cuda())
    finally:
        moe.moe_decode_step_chain_variant(0)


@pytest.mark.parametrize("name", ["35b", "35b-K2", "35b-K8", "8b", "tiny"])
def test_chain_kernels_are_coresident(name):
    """The chained step relies on a CTA of kernel A(N+1) sitting on an SM
    beside one of B(N), so that A(N+1) copies its weights while B(N) runs: a
    register spill or a shared-memory change that broke this would only show
    as a slower step.  The library's residency query checks it on the
    device (occupancy API, shared memory incl. reservations, registers)."""
    from int4_expert_gemv_gb300 import moe
    from int4_expert_gemv_gb300.model import DecodeStack, DeviceModel
    cfg = ALL[name] if name == "tiny" else replace(ALL[name], L=1)
    st = DecodeStack(DeviceModel(cfg), fused="chain")
    info = moe.moe_decode_step_chain_info(st.sd)
    assert info["local_bytes_a"] == 0 and info["local_bytes_b"] == 0, info
    assert info["regs_a"] <= 64 and info["regs_b"] <= 64, info
    assert info["ctas_a"] >= 1 and info["ctas_b"] >= 1, info
    assert info["coresident"] == 1, info
