"""Pins of the CPU oracle against things other than itself.

Each test checks one oracle function against a closed form, a value printed
on the pages, a library routine, brute force, or an invariant the definition
implies.  None of these tests needs a GPU.
"""
import itertools
from dataclasses import replace
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from int4_expert_gemv_gb300 import synth
from int4_expert_gemv_gb300.configs import TINY

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_values(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split("=")
            vals[k.strip()] = float(v)
    return vals


# --------------------------------------------------------------- fp16 / bf16
def test_f16_widening_matches_numpy_for_every_pattern(orc):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([orc.f16_to_f64(int(p)) for p in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f16_round_trip_every_pattern(orc):
    for p in range(65536):
        v = orc.f16_to_f64(p)
        if math.isnan(v):
            continue
        assert orc.f64_to_f16(v) == p, hex(p)


def test_f16_ties_to_even_by_hand(orc):
    one = 0x3C00
    assert orc.f64_to_f16(1 + 2 ** -11) == one            # tie -> even (1.0)
    assert orc.f64_to_f16(1 + 3 * 2 ** -11) == one + 2    # tie -> even (odd+1)
    assert orc.f64_to_f16(1 + 2 ** -11 + 2 ** -40) == one + 1
    assert orc.f64_to_f16(2 ** -25) == 0                  # tie between 0 and 2^-24
    assert orc.f64_to_f16(3 * 2 ** -25) == 2
    assert orc.f64_to_f16(65519.99) == 0x7BFF
    assert orc.f64_to_f16(65520.0) == 0x7C00
    assert orc.f64_to_f16(-2.0) == 0xC000


def test_f16_rounding_matches_numpy_on_random_doubles(orc):
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.normal(0, 1, 3000), rng.normal(0, 1e-5, 1000),
                        rng.normal(0, 3e4, 500)])
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    got = np.array([orc.f64_to_f16(float(x)) for x in v], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_round_trip_every_pattern(orc):
    for p in range(65536):
        v = orc.bf16_to_f64(p)
        if math.isnan(v):
            continue
        assert orc.f64_to_bf16(v) == p, hex(p)


def test_bf16_rounding_matches_torch_on_float32_values(orc):
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.normal(0, 1, 3000), rng.normal(0, 1e-30, 300)]).astype(np.float32)
    # make some exact ties: values halfway between two bf16 neighbours
    ties = (np.arange(1, 200, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    v = np.concatenate([v, ties[np.isfinite(ties)]])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.f64_to_bf16(float(x)) for x in v], dtype=np.uint16)
    assert np.array_equal(got, ref)


# --------------------------------------------------------------- decode
def _fixture_words():
    rows = []
    for line in open(os.path.join(GOLDEN, "packed_words.txt")):
        line = line.split("#")[0].strip()
        if line:
            parts = line.split()
            rows.append((int(parts[0]), int(parts[1], 16), [int(x) for x in parts[2:]]))
    return rows


@pytest.mark.parametrize("scale,bias", [(0.5, -1.0), (0.0078125, 0.125), (0.0, -0.25)])
def test_decode_fixture_words(orc, scale, bias):
    s16 = np.float16(scale).view(np.uint16)
    b16 = np.float16(bias).view(np.uint16)
    for bits, word, ns in _fixture_words():
        per = 32 // bits
        cols = 64                       # one group: the word repeated
        q = np.full((1, cols // per), word, np.uint32)
        m = dict(q=q, s=np.array([[s16]]), b=np.array([[b16]]), rows=1, cols=cols,
                 bits=bits, group=64)
        for k in range(per):
            assert orc.weight(m, 0, k) == ns[k] * scale + bias


@pytest.mark.parametrize("bits", [4, 2])
def test_decode_every_value_at_every_position(orc, bits):
    per = 32 // bits
    s, b = 0.375, -2.5
    for v in range(1 << bits):
        for j in range(per):
            q = np.zeros((1, 64 // per), np.uint32)
            q[0, 1] = np.uint32(v << (bits * j))
            m = dict(q=q, s=np.full((1, 1), np.float16(s).view(np.uint16)),
                     b=np.full((1, 1), np.float16(b).view(np.uint16)),
                     rows=1, cols=64, bits=bits, group=64)
            w = orc.dequant(m)[0]
            expect = np.full(64, b)
            expect[per + j] = v * s + b
            assert np.array_equal(w, expect)


def test_decode_uses_the_group_of_each_column(orc):
    rows, cols = 3, 256
    rng = np.random.default_rng(2)
    q = rng.integers(0, 2 ** 32, size=(rows, cols // 8), dtype=np.uint64).astype(np.uint32)
    s = rng.normal(0, 0.01, (rows, cols // 64)).astype(np.float16)
    b = rng.normal(0, 0.05, (rows, cols // 64)).astype(np.float16)
    m = dict(q=q, s=s.view(np.uint16), b=b.view(np.uint16), rows=rows, cols=cols, bits=4, group=64)
    w = orc.dequant(m)
    n = synth.unpack(q, 4).astype(np.float64)
    for o in range(rows):
        for k in range(cols):
            assert w[o, k] == n[o, k] * float(s[o, k // 64]) + float(b[o, k // 64])


# --------------------------------------------------------------- GEMV
def _rand_affine(rows, cols, bits, seed):
    return synth.affine(seed, 7, rows, cols, bits, 0.02)


@pytest.mark.parametrize("bits", [4, 2])
def test_gemv_equals_dense_matmul(orc, bits):
    m = _rand_affine(48, 320, bits, 3)
    x = np.random.default_rng(4).normal(size=320)
    y = orc.gemv(m, x)
    ref = orc.dequant(m) @ x
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)


def test_gemv_unit_vectors_give_columns(orc):
    m = _rand_affine(16, 128, 4, 5)
    w = orc.dequant(m)
    for k in (0, 1, 7, 8, 63, 64, 127):
        e = np.zeros(128)
        e[k] = 1.0
        assert np.array_equal(orc.gemv(m, e), w[:, k])


def test_gemv_fma_form_identity(orc):
    """sum_k fma(n, s*x, b*x) equals sum_k (n*s + b)*x (the pages' FMA form)."""
    g = _golden_values("page_values.txt")
    n, s, b, x = g["fma_form.nibble"], g["fma_form.scale"], g["fma_form.bias"], g["fma_form.x"]
    assert n * (s * x) + b * x == g["fma_form.value"] == (n * s + b) * x
    m = _rand_affine(8, 192, 4, 6)
    xs = np.random.default_rng(7).normal(size=192)
    nq = synth.unpack(m["q"], 4).astype(np.float64)
    sc = m["s"].view(np.float16).astype(np.float64)
    bi = m["b"].view(np.float16).astype(np.float64)
    fma_form = np.array([sum(nq[o, k] * (sc[o, k // 64] * xs[k]) + bi[o, k // 64] * xs[k]
                             for k in range(192)) for o in range(8)])
    assert np.allclose(orc.gemv(m, xs), fma_form, rtol=1e-12, atol=1e-14)


def test_quantiser_error_bound(orc):
    """Generator + oracle decode: every decoded weight lies within half a
    quantisation step (plus the fp16 rounding of scale and bias) of w."""
    w = synth.gauss(9, 11, (64, 512), 0.02)
    for bits in (4, 2):
        q, s, b = synth.quantize(w, bits)
        m = dict(q=q, s=s, b=b, rows=64, cols=512, bits=bits, group=64)
        wd = orc.dequant(m)
        lv = (1 << bits) - 1
        wg = w.astype(np.float64).reshape(64, 8, 64)
        s32 = (wg.max(2) - wg.min(2)) / lv
        sf = s.view(np.float16).astype(np.float64)
        bf = b.view(np.float16).astype(np.float64)
        bound = 0.5 * sf + np.abs(bf - wg.min(2)) + lv * np.abs(sf - s32) + 1e-7
        err = np.abs(wd.reshape(64, 8, 64) - wg).max(2)
        assert (err <= bound).all()


# --------------------------------------------------------------- LoRA
def _lora(r, din, dout, seed, scale=2.0, zero_b=False):
    A = synth.gauss_f16(seed, 1, (r, din), 0.01)
    B = np.zeros((dout, r), np.uint16) if zero_b else synth.gauss_f16(seed, 2, (dout, r), 0.01)
    return dict(A=A, B=B, scale=scale)


def test_lora_zero_b_is_identity(orc):
    x = np.random.default_rng(8).normal(size=64)
    y = np.random.default_rng(9).normal(size=32)
    assert np.array_equal(orc.lora_apply(_lora(8, 64, 32, 1, zero_b=True), x, y), y)


def test_lora_equals_merged_dense(orc):
    m = _rand_affine(32, 128, 4, 10)
    l = _lora(8, 128, 32, 2, scale=16 / 8)
    x = np.random.default_rng(11).normal(size=128)
    got = orc.lora_apply(l, x, orc.gemv(m, x))
    A = l["A"].view(np.float16).astype(np.float64)
    B = l["B"].view(np.float16).astype(np.float64)
    merged = orc.dequant(m) + l["scale"] * (B @ A)
    assert np.allclose(got, merged @ x, rtol=1e-12, atol=1e-14)


# --------------------------------------------------------------- activations
def test_gelu_closed_forms(orc):
    assert orc.gelu_erf(0.0) == 0.0
    assert abs(orc.gelu_erf(1.0) - 0.8413447460685429) < 1e-15   # Phi(1)
    for a in np.linspace(-6, 6, 61):
        assert abs(orc.gelu_erf(a) - orc.gelu_erf(-a) - a) < 1e-14
        ref = 0.5 * a * (1 + scipy.special.erf(a / math.sqrt(2)))
        assert abs(orc.gelu_erf(a) - ref) < 1e-15


def test_silu_closed_forms(orc):
    assert orc.silu(0.0) == 0.0
    assert abs(orc.silu(1.0) - 0.7310585786300049) < 1e-15     # 1/(1+e^-1)
    for a in np.linspace(-20, 20, 81):
        assert abs(orc.silu(a) - orc.silu(-a) - a) < 1e-13
        assert abs(orc.silu(a) - a * scipy.special.expit(a)) < 1e-14


# --------------------------------------------------------------- top-K
def test_topk_brute_force_subsets(orc):
    rng = np.random.default_rng(12)
    for E in (4, 7, 12):
        for K in range(1, E):
            z = rng.normal(size=E)
            best = max(itertools.combinations(range(E), K), key=lambda c: sum(z[list(c)]))
            idx, w, margin = orc.topk(z, K)
            assert set(idx.tolist()) == set(best)
            zs = np.sort(z)[::-1]
            assert margin == zs[K - 1] - zs[K]


def test_topk_order_and_ties_match_sorted(orc):
    rng = np.random.default_rng(13)
    for trial in range(200):
        E = int(rng.integers(2, 80))
        K = int(rng.integers(1, min(E, 9) + 1))
        z = rng.integers(-3, 4, size=E).astype(np.float64) * 0.5   # many ties
        ref = sorted(range(E), key=lambda e: (-z[e], e))[:K]
        idx, w, margin = orc.topk(z, K)
        assert idx.tolist() == ref
        if K < E:
            srt = sorted(z, reverse=True)
            assert margin == srt[K - 1] - srt[K]
        else:
            assert margin == math.inf


def test_route_weights_invariants(orc):
    rng = np.random.default_rng(14)
    for E, K in ((16, 2), (256, 4), (256, 8), (512, 4)):
        z = rng.normal(size=E)
        idx, w, _ = orc.topk(z, K)
        assert abs(w.sum() - 1.0) < 1e-12
        assert (np.diff(w) <= 0).all()                       # same order as z
        for a in range(K):
            for b in range(K):
                assert abs(w[a] / w[b] - math.exp(z[idx[a]] - z[idx[b]])) < 1e-9
    idx, w, _ = orc.topk(rng.normal(size=9), 1)
    assert w.tolist() == [1.0]


# --------------------------------------------------------------- combine
def test_combine_closed_forms(orc):
    rng = np.random.default_rng(15)
    d, K = 64, 3
    res = rng.normal(size=d)
    w = np.array([0.5, 0.3, 0.2])
    zero = np.zeros((K + 1, d))
    out, xn = orc.combine(zero, w, True, res)
    assert np.array_equal(out, res)
    ms = np.mean(res ** 2)
    assert abs(np.mean(xn ** 2) - ms / (ms + 1e-6)) < 1e-12
    y = rng.normal(size=(K + 1, d))
    out, _ = orc.combine(y, w, True, res)
    assert np.allclose(out, res + w @ y[:K] + y[K], rtol=1e-14, atol=1e-14)
    out2, _ = orc.combine(y[:K], w, False, res)
    assert np.allclose(out2, res + w @ y[:K], rtol=1e-14, atol=1e-14)


# --------------------------------------------------------------- head
def _head(E=16, d=64, H=64, seed=21):
    cfg = TINY.__class__(**{**TINY.__dict__, "E": E, "d": d, "H": H, "seed": seed})
    return cfg, synth.head_host(cfg, 0)


def test_head_feature_width_matches_the_page(orc):
    g = _golden_values("page_values.txt")
    d, E = int(g["head_input_width.d_model"]), int(g["head_input_width.E"])
    f = orc.head_features(d, E, np.zeros(d), np.array([1, 5, 9, 200]),
                          np.array([0, 2, 4, 255]), 4)
    assert f.shape[0] == g["head_input_width.value"]
    assert f[d:].sum() == 8 and f[d + 1] == 1 and f[d + E + 255] == 1


def test_head_with_zero_mlp_is_its_linear_path(orc):
    cfg, hd = _head()
    x = np.random.default_rng(16).normal(size=cfg.d)
    cur, prev = np.array([3, 7]), np.array([1, 7])
    zero_mlp = dict(hd)
    for k in ("fc1x", "fc2"):
        m = dict(hd[k])
        m["s"] = np.zeros_like(m["s"])
        m["b"] = np.zeros_like(m["b"])
        zero_mlp[k] = m
    zero_mlp["fc1_tab"] = np.zeros_like(hd["fc1_tab"])
    zero_mlp["b1"] = np.zeros_like(hd["b1"])
    zero_mlp["b2"] = np.zeros_like(hd["b2"])
    z = orc.head_logits(zero_mlp, x, cur, prev, 2)
    f = orc.head_features(cfg.d, cfg.E, x, cur, prev, 2)
    lfull = np.concatenate([orc.dequant(hd["lx"]),
                            hd["l_tab"].view(np.float16).astype(np.float64).T], axis=1)
    ref = lfull @ f + hd["bl"].view(np.float16).astype(np.float64)
    assert np.allclose(z, ref, rtol=1e-12, atol=1e-13)


def test_head_without_tables_is_the_plain_router(orc):
    cfg, hd = _head()
    router = synth.router_host(cfg, 0)
    x = np.random.default_rng(17).normal(size=cfg.d)
    z_router = orc.head_logits(router, x)
    assert np.allclose(z_router, orc.gemv(router["lx"], x), rtol=1e-13, atol=1e-14)
    # the l path of head 0 starts from the target layer's router (same tensor)
    assert np.array_equal(hd["lx"]["q"], synth.router_host(cfg, synth.head_target(cfg, 0))["lx"]["q"])


def test_head_one_hot_terms_equal_table_rows(orc):
    cfg, hd = _head()
    rng = np.random.default_rng(18)
    x = rng.normal(size=cfg.d)
    cur, prev = np.array([2, 11]), np.array([11, 0])
    z = orc.head_logits(hd, x, cur, prev, 2)
    t1 = hd["fc1_tab"].view(np.float16).astype(np.float64)
    tl = hd["l_tab"].view(np.float16).astype(np.float64)
    f16 = lambda a: a.view(np.float16).astype(np.float64)
    a = orc.gemv(hd["fc1x"], x) + t1[cur].sum(0) + t1[cfg.E + prev].sum(0) + f16(hd["b1"])
    g = 0.5 * a * (1 + scipy.special.erf(a / math.sqrt(2)))
    ref = (orc.dequant(hd["fc2"]) @ g + f16(hd["b2"]) + orc.gemv(hd["lx"], x)
           + tl[cur].sum(0) + tl[cfg.E + prev].sum(0) + f16(hd["bl"]))
    assert np.allclose(z, ref, rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------- experts
def test_expert_forward_matches_dense_composition(orc):
    ex = synth.expert_host(TINY, 0, 5)
    x = np.random.default_rng(19).normal(size=TINY.d)
    h, y = orc.expert_forward(ex, x)
    g = orc.dequant(ex["gate"]) @ x
    u = orc.dequant(ex["up"]) @ x
    hh = g * scipy.special.expit(g) * u
    l = ex["lora_down"]
    A = l["A"].view(np.float16).astype(np.float64)
    B = l["B"].view(np.float16).astype(np.float64)
    yy = (orc.dequant(ex["down"]) + l["scale"] * B @ A) @ hh
    assert np.allclose(h, hh, rtol=1e-11, atol=1e-13)
    assert np.allclose(y, yy, rtol=1e-11, atol=1e-13)


def test_expert_with_zero_gate_outputs_zero(orc):
    ex = synth.expert_host(TINY, 0, 6)
    for k in ("s", "b"):
        ex["gate"][k] = np.zeros_like(ex["gate"][k])
    h, y = orc.expert_forward(ex, np.ones(TINY.d))
    assert not h.any() and not y.any()


def test_expert_h_rounding_to_bf16(orc):
    ex = synth.expert_host(TINY, 0, 7)
    x = np.random.default_rng(20).normal(size=TINY.d)
    h, _ = orc.expert_forward(ex, x, round_h_bf16=False)
    hb, _ = orc.expert_forward(ex, x, round_h_bf16=True)
    ref = torch.from_numpy(h).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    # h is not float32-exact, so compare through double -> bf16 directly
    direct = np.array([orc.bf16_to_f64(orc.f64_to_bf16(v)) for v in h])
    assert np.array_equal(hb, direct)
    assert np.abs(hb - ref).max() <= np.abs(h).max() * 2 ** -8


def test_expert_ffn_slots(orc):
    exps = [synth.expert_host(TINY, 0, e) for e in range(TINY.E)]
    sh = synth.expert_host(TINY, 0, synth.SHARED_EXPERT)
    x = np.random.default_rng(21).normal(size=(3, TINY.d))
    idx = np.array([[1, 4], [15, 0], [4, 4]], np.int32)
    y = orc.expert_ffn(exps, sh, x, idx)
    assert y.shape == (3, 3, TINY.d)
    for t in range(3):
        for k in range(2):
            assert np.array_equal(y[t, k], orc.expert_forward(exps[idx[t, k]], x[t])[1])
        assert np.array_equal(y[t, 2], orc.expert_forward(sh, x[t])[1])


# --------------------------------------------------------------- stack
def _tiny_layers(cfg):
    return [dict(experts=[synth.expert_host(cfg, 0, e) for e in range(cfg.E)],
                 shared=None, router=synth.router_host(cfg, 0),
                 head=synth.head_host(cfg, 0))]


def test_single_layer_stack_follows_its_own_prediction(orc):
    """Tiny stack: step 0 routes with the router; step t>0 uses the head's
    top-K from step t-1 (fed cur = route at t-1, prev = route at t-2)."""
    cfg = TINY
    layers = _tiny_layers(cfg)
    run = orc.StackRunner(layers, cfg.d, cfg.E, cfg.K, single_layer_self_predict=True)
    ly = layers[0]
    prev_route, pred = None, None
    for t in range(4):
        x0 = synth.step_input(cfg, t)[0].astype(np.float64)
        r = run.step(x0)
        if t == 0:
            z = orc.head_logits(ly["router"], x0)
        else:
            z = pred_z
        idx, w, margin = orc.topk(z, cfg.K)
        assert r["idx"][0].tolist() == idx.tolist()
        assert np.allclose(r["w"][0], w, rtol=1e-14)
        y = orc.expert_ffn(ly["experts"], None, x0[None], idx[None])[0]
        out, _ = orc.combine(y, w, False, x0)
        assert np.allclose(r["out"], out, rtol=1e-13, atol=1e-13)
        pred_z = orc.head_logits(ly["head"], x0, idx, prev_route, cfg.K)
        prev_route = idx


def test_stack_teacher_forcing_only_at_near_ties(orc):
    cfg = TINY
    run = orc.StackRunner(_tiny_layers(cfg), cfg.d, cfg.E, cfg.K, single_layer_self_predict=True)
    x0 = synth.step_input(cfg, 0)[0]
    own = run.step(x0)
    run2 = orc.StackRunner(_tiny_layers(cfg), cfg.d, cfg.E, cfg.K, single_layer_self_predict=True)
    other = np.array([[0, 1]], np.int32)
    # margin above the threshold: the external route is ignored
    r = run2.step(x0, ext_idx=other, tie_margin=-1.0)
    assert r["idx"].tolist() == own["idx"].tolist() and not r["forced"].any()
    # threshold above the margin: the external route is adopted, weights recomputed
    run3 = orc.StackRunner(_tiny_layers(cfg), cfg.d, cfg.E, cfg.K, single_layer_self_predict=True)
    r = run3.step(x0, ext_idx=other, tie_margin=1e9)
    assert r["idx"].tolist() == other.tolist() and r["forced"].all()
    assert abs(r["w"].sum() - 1) < 1e-12


# --------------------------------------------------------------- LoRA merge
def _codes(m):
    return synth.unpack(np.asarray(m["q"]), m["bits"])


@pytest.mark.parametrize("bits", [4, 2])
def test_merge_without_adapter_is_idempotent(orc, bits):
    """Requantising weights that came out of the min/max quantiser returns
    them unchanged wherever a group holds both extreme codes (then lo = b and
    hi = b + (2^bits - 1) s exactly, so s' = s, b' = b and q' = q)."""
    m = synth.affine(21, 3, 48, 256, bits, 0.02)
    got = orc.merge_lora(m, None)
    qmax = (1 << bits) - 1
    q, q2 = _codes(m).reshape(48, 4, 64), _codes(got).reshape(48, 4, 64)
    full = (q.min(2) == 0) & (q.max(2) == qmax)
    assert full.mean() > 0.9
    assert np.array_equal(q2[full], q[full])
    assert np.array_equal(got["s"][full], np.asarray(m["s"])[full])
    assert np.array_equal(got["b"][full], np.asarray(m["b"])[full])


def test_merge_exact_steps_and_sub_step_delta(orc):
    """Deltas that are whole quantisation steps move the bias and keep every
    code; a sub-step delta on one interior weight is lost entirely.  Row 0
    gains one step (B[0][0] A[0] = s_0), row 2 two steps (B[2][1] A[1] =
    2 s_2), row 1 gets 0.3 s_1 on one interior weight (B[1][2] A[2]).  A
    transposed operand or a swapped index moves the wrong row."""
    m = synth.affine(22, 4, 3, 128, 4, 0.02)
    s = np.asarray(m["s"]).view(np.float16).astype(np.float64)
    b = np.asarray(m["b"]).view(np.float16).astype(np.float64)
    q = _codes(m)
    k1 = next(k for k in range(128) if 2 <= q[1, k] <= 13)
    A = np.zeros((3, 128), np.float64)
    A[0] = np.repeat(s[0], 64)
    A[1] = np.repeat(2 * s[2], 64)
    A[2, k1] = 0.3 * s[1, k1 // 64]
    B = np.zeros((3, 3), np.float64)
    B[0, 0] = B[2, 1] = B[1, 2] = 1.0
    l = dict(A=A.astype(np.float16).view(np.uint16), B=B.astype(np.float16).view(np.uint16),
             scale=1.0)
    assert np.array_equal(l["A"].view(np.float16).astype(np.float64)[:2], A[:2])   # exact in fp16
    got = orc.merge_lora(m, l)
    assert np.array_equal(_codes(got), q)
    assert np.array_equal(got["s"], np.asarray(m["s"]))
    f16 = lambda v: np.float16(v).view(np.uint16)
    for g in range(2):
        assert got["b"][0, g] == f16(b[0, g] + s[0, g])
        assert got["b"][1, g] == m["b"][1, g]
        assert got["b"][2, g] == f16(b[2, g] + 2 * s[2, g])


@pytest.mark.parametrize("bits", [4, 2])
def test_merge_error_bound(orc, bits):
    """Every merged weight lies within half a new quantisation step (plus the
    fp16 rounding of the new scale and bias and the binary32 arithmetic) of
    the exact W + scale B A, computed densely in fp64 with a library matmul."""
    m = synth.affine(23, 5, 32, 256, bits, 0.02)
    l = _lora(16, 256, 32, 7, scale=2.0)
    got = orc.merge_lora(m, l)
    A = l["A"].view(np.float16).astype(np.float64)
    B = l["B"].view(np.float16).astype(np.float64)
    exact = (orc.dequant(m) + l["scale"] * (B @ A)).reshape(32, 4, 64)
    wd = orc.dequant(got).reshape(32, 4, 64)
    qmax = (1 << bits) - 1
    s2 = got["s"].view(np.float16).astype(np.float64)
    b2 = got["b"].view(np.float16).astype(np.float64)
    span = (exact.max(2) - exact.min(2)) / qmax
    bound = 0.5 * s2 + np.abs(b2 - exact.min(2)) + qmax * np.abs(s2 - span) + 1e-6
    assert (np.abs(wd - exact).max(2) <= bound).all()


@pytest.mark.parametrize("bits", [4, 2])
def test_merge_comparison_tolerates_only_boundary_decisions(orc, bits):
    """The GPU-merge comparison (tests/_util.py) accepts the oracle's own
    output and a binary32 evaluation of the same merge (numpy float32, no
    fused operations), and rejects a code, a scale or a bias moved away from
    a rounding boundary."""
    from _util import assert_merge_matches
    m = synth.affine(24, 6, 40, 256, bits, 0.02)
    l = _lora(17, 256, 40, 16, scale=2.0)
    ref = orc.merge_lora(m, l)
    assert assert_merge_matches(orc, ref, ref["q"], ref["s"], ref["b"], "self") == 0
    # binary32: w = q s + b + scale (B A), min/max, fp16 rounding, codes
    f32 = np.float32
    A = l["A"].view(np.float16).astype(f32)
    B = l["B"].view(np.float16).astype(f32)
    qn = _codes(m).astype(f32)
    s = np.repeat(np.asarray(m["s"]).view(np.float16).astype(f32), 64, axis=1)
    b = np.repeat(np.asarray(m["b"]).view(np.float16).astype(f32), 64, axis=1)
    w = (qn * s + b) + f32(2.0) * (B @ A)
    wg = w.reshape(40, 4, 64)
    qmax = f32((1 << bits) - 1)
    s2 = ((wg.max(2) - wg.min(2)) / qmax).astype(np.float16)
    b2 = wg.min(2).astype(np.float16)
    s2f = np.repeat(s2.astype(f32), 64, axis=1)
    b2f = np.repeat(b2.astype(f32), 64, axis=1)
    codes = np.clip(np.rint((w - b2f) / s2f), 0, qmax).astype(np.uint32)
    per = 32 // bits
    q32 = (codes.reshape(40, -1, per) << (bits * np.arange(per, dtype=np.uint32))).sum(2).astype(np.uint32)
    assert_merge_matches(orc, ref, q32, s2.view(np.uint16), b2.view(np.uint16), "binary32")
    # planted mistakes (in copies of the oracle's output): each is caught
    t = ref["t_pre"]
    k = int(np.argmin(np.abs(np.abs(t - np.floor(t) - 0.5) - 0.25)))     # far from a midpoint
    o, c = divmod(k, 256)
    q_bad = ref["q"].copy()
    q_bad[o, c // per] ^= np.uint32(1 << (bits * (c % per)))
    with pytest.raises(AssertionError):
        assert_merge_matches(orc, ref, q_bad, ref["s"], ref["b"], "code")
    s_bad = ref["s"].copy()
    s_bad[3, 1] += 1
    with pytest.raises(AssertionError):
        assert_merge_matches(orc, ref, ref["q"], s_bad, ref["b"], "scale")
    b_bad = ref["b"].copy()
    b_bad[5, 2] += 2
    with pytest.raises(AssertionError):
        assert_merge_matches(orc, ref, ref["q"], ref["s"], b_bad, "bias")


def test_multi_layer_stack_routes_from_the_previous_layers_head(orc):
    """A 3-layer stack (tiny shapes, shared expert) over 4 steps, rebuilt from
    the separately pinned functions: layer 0 routes with its own router every
    step; layer N >= 1 routes with its own router at t = 0 and afterwards with
    the top-K head N-1 computed at t-1; head N runs on x_N with cur = layer
    N's route at t and prev = layer N's route at t-1, and x_{N+1} is the RMS of
    out_N.  Applying head N's prediction to layer N instead of N+1, or taking
    prev from another layer, changes the routes and fails this test."""
    cfg = replace(TINY, L=3, depth=3, self_predict=False)
    L = cfg.L
    layers = [dict(experts=[synth.expert_host(cfg, n, e) for e in range(cfg.E)],
                   shared=synth.expert_host(cfg, n, synth.SHARED_EXPERT),
                   router=synth.router_host(cfg, n), head=synth.head_host(cfg, n))
              for n in range(L)]
    run = orc.StackRunner(layers, cfg.d, cfg.E, cfg.K)
    pred_z = [None] * L          # logits head N-1 gave for layer N at the last step
    prev = [None] * L            # route layer N used at the last step
    seen = set()
    for t in range(4):
        x0 = synth.step_input(cfg, t)[0].astype(np.float64)
        r = run.step(x0)
        stream, x = x0, x0
        cur, nxt = [None] * L, [None] * L
        for N in range(L):
            ly = layers[N]
            z = orc.head_logits(ly["router"], x) if (N == 0 or t == 0) else pred_z[N]
            idx, w, _ = orc.topk(z, cfg.K)
            assert r["idx"][N].tolist() == idx.tolist(), (t, N)
            assert np.array_equal(r["w"][N], w), (t, N)
            y = orc.expert_ffn(ly["experts"], ly["shared"], x[None], idx[None])[0]
            out, xn = orc.combine(y, w, True, stream)
            if N + 1 < L:
                nxt[N + 1] = orc.head_logits(ly["head"], x, idx, prev[N], cfg.K)
            cur[N] = idx
            seen.add(tuple(idx.tolist()))
            stream, x = out, xn
        assert np.array_equal(r["out"], stream), t
        prev, pred_z = cur, nxt
    assert len(seen) > 6          # the routes do change from layer to layer and step to step


# --------------------------------------------------------------- threads
def test_threaded_rows_give_the_same_bits(orc):
    """The CPU baseline times the oracle at several thread counts: a row is
    still one thread's ascending-order sum, so GEMV and head logits are the
    same bits at 1 and 4 threads."""
    m = _rand_affine(96, 512, 4, 31)
    x = np.random.default_rng(32).normal(size=512)
    cfg, hd = _head(E=32, d=128, H=64, seed=33)
    xh = np.random.default_rng(34).normal(size=cfg.d)
    cur, prev = np.array([3, 7]), np.array([1, 30])
    try:
        orc.set_threads(1)
        y1, z1 = orc.gemv(m, x), orc.head_logits(hd, xh, cur, prev, 2)
        orc.set_threads(4)
        y4, z4 = orc.gemv(m, x), orc.head_logits(hd, xh, cur, prev, 2)
    finally:
        orc.set_threads(1)
    assert np.array_equal(y1, y4) and np.array_equal(z1, z4)
