"""Predicted routes against the layers' own routers (the prediction-mismatch
measurement): the own-router top-K the GPU computes on each layer's input
matches the oracle's router on the same input (as index sets, where the
oracle's margin clears the tie bar), and the agreement statistics are
consistent with the routes they are computed from."""
import numpy as np
import pytest
import torch

import oracle as orc
from int4_expert_gemv_gb300 import synth
from int4_expert_gemv_gb300.configs import ALL, TINY
from _util import TIE

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    from int4_expert_gemv_gb300 import build
    build.build()
    from int4_expert_gemv_gb300 import moe
    moe.lib()
    synth._gpu()
    return moe


@pytest.mark.parametrize("name", ["tiny", "35b-L4"])
def test_own_routes_match_the_oracle_router(m, name):
    from int4_expert_gemv_gb300.model import DecodeStack, DeviceModel
    cfg = TINY if name == "tiny" else ALL[name]
    dm = DeviceModel(cfg)
    st = DecodeStack(dm)
    checked = 0
    for t in range(3):
        st.step(torch.from_numpy(synth.step_input(cfg, t)[0]).cuda())
        if t == 0:
            continue
        own, mg = st.own_routes(t)
        own = own.cpu().numpy()
        xs = st.xs.cpu().double().numpy()
        for N in range(cfg.depth):
            z = orc.head_logits(synth.router_host(cfg, N % cfg.L), xs[N])
            idx, _, margin = orc.topk(z, cfg.K)
            if margin > TIE:
                assert set(own[N].tolist()) == set(idx.tolist()), (t, N)
                checked += 1
    assert checked >= cfg.depth


def test_prediction_agreement_statistics(m):
    from int4_expert_gemv_gb300.model import DeviceModel, prediction_agreement
    cfg = ALL["35b-L4"]
    res = prediction_agreement(DeviceModel(cfg), steps=4)
    assert res["layer_steps"] == 4 * (cfg.depth - 1)
    assert 0.0 <= res["equal_sets"] <= res["mean_overlap"] <= 1.0
    assert res["chance_overlap"] == cfg.K / cfg.E
