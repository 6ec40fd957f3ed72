"""Helpers shared by the GPU parity tests (no test functions here)."""
from __future__ import annotations

import numpy as np

from int4_expert_gemv_gb300 import synth

TOL = 2e-3      # max |got - ref| <= TOL * rms(ref), per output tensor
TIE = 1e-4      # route indices are compared where the oracle margin exceeds this


def rms(a) -> float:
    a = np.asarray(a, dtype=np.float64)
    return float(np.sqrt(np.mean(a * a)))


def assert_close(got, ref, what: str, tol: float = TOL):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = float(np.abs(got - ref).max())
    bound = tol * rms(ref)
    assert err <= bound, f"{what}: max|err| {err:.3e} > {tol}*rms(ref) = {bound:.3e}"
    return err / max(rms(ref), 1e-300)


def bf16_h_allowance(ex: dict, x) -> np.ndarray:
    """Per-output allowance for the bf16 rounding of h (the batched path's
    activations).  The GPU decides that rounding from an fp32 h, the oracle
    from an fp64 one: where the oracle's h lies within 1e-5 relative of a
    midpoint between two bf16 neighbours, either neighbour is a correct
    rounding.  For those f the output may move by the effective down column
    (W_d plus the scaled LoRA product) times the neighbours' gap; the sum of
    those moves bounds the extra difference."""
    import oracle as orc
    h, _ = orc.expert_forward(ex, x, round_h_bf16=False)
    lo_bits = h.astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    lo = lo_bits.view(np.float32).astype(np.float64)
    hi = (lo_bits + np.uint32(0x10000)).view(np.float32).astype(np.float64)
    amb = np.abs(h - 0.5 * (lo + hi)) <= 1e-5 * np.abs(h)
    d = ex["down"]["rows"]
    if not amb.any():
        return np.zeros(d)
    W = orc.dequant(ex["down"])
    if "lora_down" in ex:
        ld = ex["lora_down"]
        A = ld["A"].view(np.float16).astype(np.float64)
        B = ld["B"].view(np.float16).astype(np.float64)
        W = W + ld["scale"] * (B @ A)
    return np.abs(W[:, amb]) @ np.abs(hi - lo)[amb]


def assert_close_bf16h(got, ref, ex: dict, x, what: str, tol: float = TOL):
    """assert_close, widened per output by bf16_h_allowance where needed."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    bound = tol * rms(ref)
    err = np.abs(got - ref)
    if float(err.max()) <= bound:
        return
    allow = bf16_h_allowance(ex, x)
    over = err - (bound + allow)
    assert float(over.max()) <= 0.0, (
        f"{what}: max|err| {float(err.max()):.3e} > {tol}*rms(ref) = {bound:.3e} "
        f"+ bf16-rounding allowance (worst excess {float(over.max()):.3e})")


def host_expert_from_gpu(cfg, layer: int, e: int) -> dict:
    """The logical tensors of one expert, drawn by the GPU twin of the
    generator and copied to the host (bit-identical to synth.expert_host)."""
    import torch
    d, F, bits = cfg.d, cfg.F, cfg.bits

    def aff(kind, rows, cols):
        q = torch.empty((rows, cols * bits // 32), dtype=torch.int32, device="cuda")
        s = torch.empty((rows, cols // 64), dtype=torch.int16, device="cuda")
        b = torch.empty_like(s)
        synth.gpu_affine(cfg.seed, synth.tag(kind, layer, e), rows, cols, bits, cfg.sigma_w, q, s, b)
        return dict(q=q.cpu().numpy().view(np.uint32), s=s.cpu().numpy().view(np.uint16),
                    b=b.cpu().numpy().view(np.uint16), rows=rows, cols=cols, bits=bits, group=64)

    ex = dict(gate=aff(synth.GATE, F, d), up=aff(synth.UP, F, d), down=aff(synth.DOWN, d, F))
    r = cfg.lora_r

    def ad(ka, kb, din, dout):
        return dict(A=synth.gauss_f16(cfg.seed, synth.tag(ka, layer, e), (r, din), cfg.sigma_lora),
                    B=synth.gauss_f16(cfg.seed, synth.tag(kb, layer, e), (dout, r), cfg.sigma_lora),
                    scale=cfg.lora_scale)

    if r and cfg.lora_on == "routed_down" and e != synth.SHARED_EXPERT:
        ex["lora_down"] = ad(synth.LORA_DOWN_A, synth.LORA_DOWN_B, F, d)
    if r and cfg.lora_on == "shared_all" and e == synth.SHARED_EXPERT:
        ex["lora_gate"] = ad(synth.LORA_GATE_A, synth.LORA_GATE_B, d, F)
        ex["lora_up"] = ad(synth.LORA_UP_A, synth.LORA_UP_B, d, F)
        ex["lora_down"] = ad(synth.LORA_DOWN_A, synth.LORA_DOWN_B, F, d)
    return ex


def zero_expert(cfg) -> dict:
    """Placeholder for experts a test never routes to (all-zero weights)."""
    d, F, bits = cfg.d, cfg.F, cfg.bits

    def z(rows, cols):
        return dict(q=np.zeros((rows, cols * bits // 32), np.uint32),
                    s=np.zeros((rows, cols // 64), np.uint16),
                    b=np.zeros((rows, cols // 64), np.uint16),
                    rows=rows, cols=cols, bits=bits, group=64)
    return dict(gate=z(F, d), up=z(F, d), down=z(d, F))


MERGE_EPS = 0.01   # a rounding decision within this fraction of a grid step of a midpoint may go either way


def _f16_pair(v):
    """fp16 neighbours (bit patterns lo <= v <= hi, as values) of fp64 values,
    and whether v lies within MERGE_EPS of a step of their midpoint."""
    v = np.asarray(v, dtype=np.float64)
    r = v.astype(np.float16)
    rv = r.astype(np.float64)
    lo = np.where(rv > v, np.nextafter(r, np.float16(-np.inf)), r)
    hi = np.where(rv < v, np.nextafter(r, np.float16(np.inf)), r)
    lv, hv = lo.astype(np.float64), hi.astype(np.float64)
    near = (hv > lv) & (np.abs(v - 0.5 * (lv + hv)) <= MERGE_EPS * (hv - lv))
    return lo.view(np.uint16), hi.view(np.uint16), near


def _codes_ok(q_got, t, bits):
    """Codes decided from the pre-rounding values t: equal to clamp(rint(t))
    except within MERGE_EPS of a midpoint, where either neighbour is taken."""
    qmax = (1 << bits) - 1
    fl = np.floor(t)
    near = np.abs(t - (fl + 0.5)) <= MERGE_EPS
    exact = np.clip(np.rint(t), 0, qmax)
    alt = np.clip(np.where(t - fl < 0.5, fl + 1, fl), 0, qmax)
    return (q_got == exact) | (near & (q_got == alt))


def assert_merge_matches(orc, ref: dict, q_got, s_got, b_got, what: str):
    """GPU merge output (logical q words, s, b bit patterns) against the
    oracle's fp64 merge (oracle.merge_lora).  The new scale and bias of a
    group are compared bit for bit, except where the oracle's value before the
    fp16 rounding lies within MERGE_EPS of a step of a midpoint (binary32
    arithmetic may then land on the other neighbour).  The codes are compared
    bit for bit against the oracle's rule applied, in fp64, under the scale
    and bias the GPU chose, except where that value before rint lies within
    MERGE_EPS of a midpoint.  Returns the number of near-boundary decisions
    that went the other way."""
    bits, group = ref["bits"], ref["group"]
    s_lo, s_hi, s_near = _f16_pair(ref["s_pre"])
    b_lo, b_hi, b_near = _f16_pair(ref["b_pre"])
    s_ok = (s_got == ref["s"]) | (s_near & ((s_got == s_lo) | (s_got == s_hi)))
    b_ok = (b_got == ref["b"]) | (b_near & ((b_got == b_lo) | (b_got == b_hi)))
    assert s_ok.all(), f"{what}: {int((~s_ok).sum())} scales differ away from a rounding boundary"
    assert b_ok.all(), f"{what}: {int((~b_ok).sum())} biases differ away from a rounding boundary"
    _, t = orc.quant_codes(ref["w"], bits, group, s_got, b_got)
    per = 32 // bits
    codes = ((np.asarray(q_got, np.uint32)[:, :, None] >> (bits * np.arange(per, dtype=np.uint32)))
             & np.uint32((1 << bits) - 1)).reshape(t.shape).astype(np.float64)
    ok = _codes_ok(codes, t, bits)
    assert ok.all(), f"{what}: {int((~ok).sum())} codes differ away from a rounding boundary"
    ref_codes = ((np.asarray(ref["q"], np.uint32)[:, :, None] >> (bits * np.arange(per, dtype=np.uint32)))
                 & np.uint32((1 << bits) - 1)).reshape(t.shape)
    return int((s_got != ref["s"]).sum() + (b_got != ref["b"]).sum() + (codes != ref_codes).sum())
