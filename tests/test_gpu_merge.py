"""LoRA merge on the GPU (moe_merge_lora) against the oracle's fp64 merge:
codes, scales and biases bit for bit except at decisions that lie within a
small fraction of a grid step of a rounding midpoint (tests/_util.py:
assert_merge_matches), in place and strided; then the retention measurement
(how much of the shared expert's adapter delta the merged int4 weights keep)
against the same measurement on the oracle."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle as orc
from int4_expert_gemv_gb300 import synth
from int4_expert_gemv_gb300.configs import ALL
from _util import assert_merge_matches, host_expert_from_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    from int4_expert_gemv_gb300 import build
    build.build()
    from int4_expert_gemv_gb300 import moe
    moe.lib()
    synth._gpu()
    return moe


def _packed(m, mat):
    """Records of a logical matrix (packed on the GPU)."""
    rows, cols, bits = mat["rows"], mat["cols"], mat["bits"]
    out = torch.zeros(m.moe_packed_matrix_bytes(rows, cols, bits), dtype=torch.uint8, device="cuda")
    dev = lambda a, t: torch.from_numpy(np.ascontiguousarray(a).view(t)).cuda()
    m.moe_pack_matrix(dev(mat["q"], np.int32), dev(mat["s"], np.int16), dev(mat["b"], np.int16),
                      rows, cols, bits, out)
    return out


def _unpacked(m, rec_bytes, rows, cols, bits, first=0, step=1):
    """Logical (q, s, b) of records first, first + step, ... of a byte tensor."""
    raw = rec_bytes.cpu().numpy()
    rb = m.moe_record_bytes(cols, bits)
    cb, ng = cols * bits // 8, cols // 64
    sel = np.stack([raw[(first + i * step) * rb:(first + i * step + 1) * rb] for i in range(rows)])
    q = np.ascontiguousarray(sel[:, :cb]).view(np.uint32)
    sb = np.ascontiguousarray(sel[:, cb:cb + 4 * ng]).view(np.uint32)
    return q, (sb & 0xffff).astype(np.uint16), (sb >> 16).astype(np.uint16)


def _lora(seed, r, din, dout):
    return dict(A=synth.gauss_f16(seed, 1, (r, din), 0.01), B=synth.gauss_f16(seed, 2, (dout, r), 0.01),
                scale=2.0)


def _merge(m, src, dst, rows, cols, bits, l, stride=None, first=0):
    rb = m.moe_record_bytes(cols, bits)
    stride = stride or rb
    A = torch.from_numpy(l["A"].view(np.int16)).cuda() if l else None
    B = torch.from_numpy(l["B"].view(np.int16)).cuda() if l else None
    m.moe_merge_lora(src.data_ptr() + first * rb, stride, rows, cols, bits, A, B,
                     l["A"].shape[0] if l else 0, l["scale"] if l else 0.0,
                     dst.data_ptr() + first * rb, stride)
    torch.cuda.synchronize()


@pytest.mark.parametrize("bits,r", [(4, 16), (2, 16), (4, 0), (4, 3)])
def test_merge_matches_oracle(m, bits, r):
    rows, cols = 96, 512
    mat = synth.affine(31, 6, rows, cols, bits, 0.02)
    l = _lora(32, r, cols, rows) if r else None
    src = _packed(m, mat)
    dst = torch.full_like(src, 0xAB)
    _merge(m, src, dst, rows, cols, bits, l)
    ref = orc.merge_lora(mat, l)
    q, s, b = _unpacked(m, dst, rows, cols, bits)
    assert_merge_matches(orc, ref, q, s, b, f"int{bits} r{r}")
    # the copy is whole records (zero padding included); in place gives the same bytes
    _merge(m, src, src, rows, cols, bits, l)
    assert torch.equal(src, dst)


def test_merge_strided_rows_leave_the_others(m):
    """Every other record (the gate rows of a gate/up section): the merged
    rows match the oracle on that sub-matrix, the rows between are untouched."""
    bits, rows, cols = 4, 64, 256
    mat = synth.affine(33, 7, 2 * rows, cols, bits, 0.02)
    src = _packed(m, mat)
    before = src.clone()
    rb = m.moe_record_bytes(cols, bits)
    l = _lora(34, 8, cols, rows)
    _merge(m, src, src, rows, cols, bits, l, stride=2 * rb, first=1)
    odd = dict(mat, q=mat["q"][1::2], s=mat["s"][1::2], b=mat["b"][1::2], rows=rows)
    ref = orc.merge_lora(odd, l)
    q, s, b = _unpacked(m, src, rows, cols, bits, first=1, step=2)
    assert_merge_matches(orc, ref, q, s, b, "odd rows")
    even = src.view(2 * rows, rb)[0::2]
    assert torch.equal(even, before.view(2 * rows, rb)[0::2])


def test_retention_matches_oracle(m):
    """The retention measurement of the 35B-like shared expert (layer 0,
    adapters on gate, up and down) through the GPU path, against the oracle
    measuring the same thing with its own merge and fp64 expert."""
    from int4_expert_gemv_gb300.model import DeviceModel, lora_merge_retention
    cfg = replace(ALL["35b"], L=1, depth=1)
    dm = DeviceModel(cfg, heads=False)
    T = 4
    got = lora_merge_retention(dm, 0, T)
    ex = host_expert_from_gpu(cfg, 0, synth.SHARED_EXPERT)
    base = dict(gate=ex["gate"], up=ex["up"], down=ex["down"])
    merged = dict(gate=orc.merge_lora(ex["gate"], ex["lora_gate"]),
                  up=orc.merge_lora(ex["up"], ex["lora_up"]),
                  down=orc.merge_lora(ex["down"], ex["lora_down"]))
    x = synth.gauss(cfg.seed, 977, (T, cfg.d), 1.0).astype(np.float64)
    yb = np.stack([orc.expert_forward(base, xi)[1] for xi in x])
    yl = np.stack([orc.expert_forward(ex, xi)[1] for xi in x])
    ym = np.stack([orc.expert_forward(merged, xi)[1] for xi in x])
    dl, dmg = yl - yb, ym - yb
    ret = float((dmg * dl).sum() / (dl * dl).sum())
    assert 0.0 < ret < 1.0
    assert abs(got["retention"] - ret) < 0.02, (got["retention"], ret)
    # the merged blob itself: every section against the oracle's merge
    blob = got["merged_blob"]
    from int4_expert_gemv_gb300.model import expert_sections
    for (off, stride, rows, cols), name in zip(expert_sections(cfg), ("gate", "up", "down")):
        rb = m.moe_record_bytes(cols, cfg.bits)
        q, s, b = _unpacked(m, blob[off:], rows, cols, cfg.bits, step=stride // rb)
        assert_merge_matches(orc, merged[name], q, s, b, name)
