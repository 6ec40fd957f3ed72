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
