"""Properties of the seeded synthetic-input generator (host twin)."""
import numpy as np

from int4_expert_gemv_gb300 import synth
from int4_expert_gemv_gb300.configs import ALL, MOE35B, TINY


def test_splitmix_reference_values():
    # SplitMix64 with state 0: the first outputs of the published generator
    # (state += golden; mix(state)).
    assert synth._mix_int(synth.GOLDEN) == 0xE220A8397B1DCDAF
    assert synth._mix_int(2 * synth.GOLDEN) == 0x6E789E6AA1B965F4
    w = synth.words(0, 0, 2)
    key = synth.stream_key(0, 0)
    assert int(w[0]) == synth._mix_int(key + synth.GOLDEN)
    assert int(w[1]) == synth._mix_int(key + 2 * synth.GOLDEN)


def test_streams_are_deterministic_and_distinct():
    a = synth.gauss(1, synth.tag(synth.GATE, 0, 3), (64, 64), 0.02)
    b = synth.gauss(1, synth.tag(synth.GATE, 0, 3), (64, 64), 0.02)
    c = synth.gauss(1, synth.tag(synth.GATE, 0, 4), (64, 64), 0.02)
    d = synth.gauss(2, synth.tag(synth.GATE, 0, 3), (64, 64), 0.02)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)


def test_gaussian_moments():
    w = synth.gauss(3, 5, (1 << 20,), 0.02).astype(np.float64)
    assert abs(w.mean()) < 1e-4
    assert abs(w.std() / 0.02 - 1) < 5e-3
    assert np.abs(w).max() <= 0.02 * 131070 / synth.IRWIN4_STD * (1 + 1e-6)
    kurt = ((w - w.mean()) ** 4).mean() / w.var() ** 2
    assert 2.6 < kurt < 3.0          # Irwin-Hall n=4: 3 - 1.2/4 = 2.7


def test_quantiser_levels_and_constant_groups():
    w = synth.gauss(4, 6, (8, 128), 0.02)
    w[0, :64] = 0.125                 # constant group: s == 0, q == 0
    for bits in (4, 2):
        q, s, b = synth.quantize(w, bits)
        n = synth.unpack(q, bits)
        assert n.max() <= (1 << bits) - 1
        assert s[0, 0] == 0 and (n[0, :64] == 0).all()
        assert b[0, 0] == np.float16(0.125).view(np.uint16)
        # every non-constant group uses both end levels (min -> 0, max -> top)
        assert (n[1:].reshape(7, 2, 64).min(2) == 0).all()


def test_pack_unpack_round_trip():
    rng = np.random.default_rng(0)
    for bits in (4, 2):
        n = rng.integers(0, 1 << bits, size=(5, 256)).astype(np.uint32)
        assert np.array_equal(synth.unpack(synth.pack(n, bits), bits), n)


def test_routes_are_k_subsets():
    r = synth.routes(4, 9, 512, 256, 4)
    assert r.shape == (512, 4)
    assert all(len(set(row)) == 4 for row in r.tolist())
    assert r.min() >= 0 and r.max() < 256
    counts = np.bincount(r.ravel(), minlength=256)
    assert counts.min() > 0           # 2048 draws over 256 experts


def test_config_expert_bytes():
    assert TINY.expert_bytes() == 55_296
    assert MOE35B.expert_bytes() == 1_769_472
    assert MOE35B.expert_bytes_per_layer() == 8_847_360
    assert ALL["wide-int4"].expert_bytes() == 7_077_888
    assert ALL["wide-int2"].expert_bytes() == 3_932_160


def test_lora_placement():
    ex = synth.expert_host(TINY, 0, 1)
    assert set(k for k in ex if k.startswith("lora")) == {"lora_down"}
    assert ex["lora_down"]["A"].shape == (8, 128) and ex["lora_down"]["B"].shape == (256, 8)
    c = MOE35B.__class__(**{**MOE35B.__dict__, "d": 128, "F": 64})
    assert not any(k.startswith("lora") for k in synth.expert_host(c, 0, 1))
    sh = synth.expert_host(c, 0, synth.SHARED_EXPERT)
    assert {k for k in sh if k.startswith("lora")} == {"lora_gate", "lora_up", "lora_down"}
