"""Seeded synthetic inputs shared by the CUDA path and the oracle.

This module produces *data* only: weights, activations and routes.  It holds
none of the layer's arithmetic (no decode, GEMV, head, top-K or combine).

Counter-based generator
-----------------------
Every tensor is identified by ``(seed, tag)``; element ``i`` draws the 64-bit
word ``mix(key + (i + 1) * GOLDEN)`` with ``key = mix(seed * GOLDEN ^ mix(tag))``,
where ``mix`` is the SplitMix64 finaliser (Steele, Lea & Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014) and ``GOLDEN`` its
increment 0x9E3779B97F4A7C15.  All arithmetic is modulo 2^64.

Gaussian values are Irwin-Hall sums of the word's four 16-bit fields,
``n = u0 + u1 + u2 + u3 - 131070`` (an exact integer), scaled once in fp32:
``w = float32(n) * float32(sigma / 37837.2272...)``.  The result is bounded at
about 3.46 sigma; its variance is sigma^2.  Because every step is an exact
integer operation or a single IEEE fp32 rounding, the CUDA twin
(``csrc/synth.cu``) reproduces it bit for bit.

Quantiser (per row, per group of 64 along the input dimension, fp32 ops):
``s = fp16((max - min) / (2^bits - 1))``, ``b = fp16(min)``,
``q = clamp(rint((w - b) / s), 0, 2^bits - 1)`` (rint ties to even; q = 0 when
s == 0).  Packing: element j of a uint32 word sits at bits ``bits*j`` (LSB
first), words row-major ``[rows][cols*bits/32]``.
"""
from __future__ import annotations

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
M64 = (1 << 64) - 1
IRWIN4_STD = float(np.sqrt(4.0 * (65536.0 ** 2 - 1.0) / 12.0))  # 37837.2272...
IRWIN4_MEAN = 131070

# tensor kinds (low bits of the tag)
GATE, UP, DOWN = 1, 2, 3
LORA_GATE_A, LORA_GATE_B, LORA_UP_A, LORA_UP_B, LORA_DOWN_A, LORA_DOWN_B = 4, 5, 6, 7, 8, 9
ROUTER = 16
FC1X, FC1_TAB, B1, FC2, B2, L_TAB, BL = 17, 18, 19, 20, 21, 22, 23
X_INPUT = 32
SHARED_EXPERT = 0xFFFFF


def tag(kind: int, layer: int = 0, expert: int = 0) -> int:
    """64-bit tensor tag: kind (8 bits) | expert (20 bits) | layer (16 bits)."""
    return ((layer & 0xFFFF) << 28) | ((expert & 0xFFFFF) << 8) | (kind & 0xFF)


def _mix_int(z: int) -> int:
    z &= M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def stream_key(seed: int, tg: int) -> int:
    return _mix_int(((seed * GOLDEN) & M64) ^ _mix_int(tg))


def _mix_np(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def words(seed: int, tg: int, n: int, start: int = 0) -> np.ndarray:
    """The n raw 64-bit words of stream (seed, tg), from element `start`."""
    key = np.uint64(stream_key(seed, tg))
    i = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix_np(key + i * np.uint64(GOLDEN))


def sigma_scale(sigma: float) -> np.float32:
    return np.float32(sigma / IRWIN4_STD)


def gauss(seed: int, tg: int, shape, sigma: float) -> np.ndarray:
    """fp32 near-Gaussian values (Irwin-Hall of 4 uniforms), exact twin of the GPU."""
    n = int(np.prod(shape))
    r = words(seed, tg, n)
    m = np.uint64(0xFFFF)
    S = ((r & m) + ((r >> np.uint64(16)) & m) + ((r >> np.uint64(32)) & m)
         + ((r >> np.uint64(48)) & m)).astype(np.int64) - IRWIN4_MEAN
    return (S.astype(np.float32) * sigma_scale(sigma)).reshape(shape)


def gauss_f16(seed: int, tg: int, shape, sigma: float) -> np.ndarray:
    """fp16 bit patterns (uint16) of gauss(), rounded to nearest even."""
    return gauss(seed, tg, shape, sigma).astype(np.float16).view(np.uint16)


def quantize(w: np.ndarray, bits: int, group: int = 64):
    """Min/max affine quantiser -> (q packed uint32, s fp16 bits, b fp16 bits)."""
    rows, cols = w.shape
    assert cols % group == 0 and bits in (2, 4)
    w = np.ascontiguousarray(w, dtype=np.float32)
    wg = w.reshape(rows, cols // group, group)
    mn = wg.min(axis=2)
    mx = wg.max(axis=2)
    levels = np.float32((1 << bits) - 1)
    s16 = ((mx - mn) / levels).astype(np.float16)
    b16 = mn.astype(np.float16)
    s = s16.astype(np.float32)[:, :, None]
    b = b16.astype(np.float32)[:, :, None]
    safe = np.where(s > 0, s, np.float32(1))
    q = np.rint((wg - b) / safe)
    q = np.where(s > 0, np.clip(q, 0, levels), 0).astype(np.uint32)
    return pack(q.reshape(rows, cols), bits), s16.view(np.uint16), b16.view(np.uint16)


def pack(q: np.ndarray, bits: int) -> np.ndarray:
    """uint32 words, element j of each word at bits bits*j (LSB first)."""
    rows, cols = q.shape
    per = 32 // bits
    q = q.astype(np.uint32).reshape(rows, cols // per, per)
    out = np.zeros((rows, cols // per), np.uint32)
    for j in range(per):
        out |= q[:, :, j] << np.uint32(bits * j)
    return out


def unpack(words_: np.ndarray, bits: int) -> np.ndarray:
    rows, nw = words_.shape
    per = 32 // bits
    out = np.zeros((rows, nw, per), np.uint32)
    for j in range(per):
        out[:, :, j] = (words_ >> np.uint32(bits * j)) & np.uint32((1 << bits) - 1)
    return out.reshape(rows, nw * per)


def affine(seed: int, tg: int, rows: int, cols: int, bits: int, sigma: float,
           group: int = 64) -> dict:
    """A quantised weight matrix as a dict {q, s, b, rows, cols, bits, group}."""
    q, s, b = quantize(gauss(seed, tg, (rows, cols), sigma), bits, group)
    return dict(q=q, s=s, b=b, rows=rows, cols=cols, bits=bits, group=group)


def routes(seed: int, tg: int, T: int, E: int, K: int) -> np.ndarray:
    """T uniform random K-subsets of range(E) (int32 [T][K]), by key order."""
    keys = words(seed, tg, T * E).reshape(T, E)
    return np.argsort(keys, axis=1, kind="stable")[:, :K].astype(np.int32)


# ------------------------------------------------------------ model tensors
def _weight(cfg, tg: int, rows: int, cols: int, prec: str, sigma: float) -> dict:
    if prec == "fp16":
        return dict(f16=gauss_f16(cfg.seed, tg, (rows, cols), sigma), rows=rows, cols=cols)
    return affine(cfg.seed, tg, rows, cols, 4 if prec == "int4" else cfg.bits, sigma, cfg.group)


def expert_host(cfg, layer: int, e: int) -> dict:
    """Logical tensors of expert e (SHARED_EXPERT for the shared one) of a
    resident layer: gate/up [F][d], down [d][F] quantised with cfg.bits, plus
    the LoRA adapters the config places on it (A [r][in], B [out][r], fp16)."""
    s, d, F, b = cfg.seed, cfg.d, cfg.F, cfg.bits
    ex = dict(gate=affine(s, tag(GATE, layer, e), F, d, b, cfg.sigma_w, cfg.group),
              up=affine(s, tag(UP, layer, e), F, d, b, cfg.sigma_w, cfg.group),
              down=affine(s, tag(DOWN, layer, e), d, F, b, cfg.sigma_w, cfg.group))
    r = cfg.lora_r

    def ad(ka, kb, din, dout):
        return dict(A=gauss_f16(s, tag(ka, layer, e), (r, din), cfg.sigma_lora),
                    B=gauss_f16(s, tag(kb, layer, e), (dout, r), cfg.sigma_lora),
                    scale=cfg.lora_scale)

    if r and cfg.lora_on == "routed_down" and e != SHARED_EXPERT:
        ex["lora_down"] = ad(LORA_DOWN_A, LORA_DOWN_B, F, d)
    if r and cfg.lora_on == "shared_all" and e == SHARED_EXPERT:
        ex["lora_gate"] = ad(LORA_GATE_A, LORA_GATE_B, d, F)
        ex["lora_up"] = ad(LORA_UP_A, LORA_UP_B, d, F)
        ex["lora_down"] = ad(LORA_DOWN_A, LORA_DOWN_B, F, d)
    return ex


def router_host(cfg, layer: int) -> dict:
    """Layer router W_r [E][d] as a head with H = 0 (logits = W_r x)."""
    return dict(d=cfg.d, E=cfg.E, H=0,
                lx=_weight(cfg, tag(ROUTER, layer), cfg.E, cfg.d, cfg.head_prec, cfg.sigma_w))


def head_target(cfg, layer: int) -> int:
    """Resident layer whose route the head of `layer` predicts."""
    return 0 if cfg.L == 1 else (layer + 1) % cfg.L


def head_host(cfg, layer: int) -> dict:
    """Prerouter head of a resident layer.  Its linear path l(x) starts from
    the target layer's router: lx is that router's tensor (same tag)."""
    s, d, E, H, p = cfg.seed, cfg.d, cfg.E, cfg.H, cfg.head_prec
    hd = dict(d=d, E=E, H=H,
              lx=_weight(cfg, tag(ROUTER, head_target(cfg, layer)), E, d, p, cfg.sigma_w),
              l_tab=gauss_f16(s, tag(L_TAB, layer), (2 * E, E), cfg.sigma_w),
              bl=gauss_f16(s, tag(BL, layer), (E,), cfg.sigma_bias))
    if H:
        hd.update(fc1x=_weight(cfg, tag(FC1X, layer), H, d, p, cfg.sigma_w),
                  fc1_tab=gauss_f16(s, tag(FC1_TAB, layer), (2 * E, H), cfg.sigma_w),
                  b1=gauss_f16(s, tag(B1, layer), (H,), cfg.sigma_bias),
                  fc2=_weight(cfg, tag(FC2, layer), E, H, p, cfg.sigma_w),
                  b2=gauss_f16(s, tag(B2, layer), (E,), cfg.sigma_bias))
    return hd


def step_input(cfg, step: int) -> np.ndarray:
    """Layer-0 hidden state of decode step `step` (fp32 [T][d], N(0,1))."""
    return gauss(cfg.seed, tag(X_INPUT, step), (cfg.T, cfg.d), 1.0)


# ------------------------------------------------------------ GPU twin
_gpu_lib = None


def _gpu():
    """libmoe_synth.so (csrc/synth.cu), the bit-exact CUDA twin of this module."""
    global _gpu_lib
    if _gpu_lib is None:
        import ctypes as C
        import os
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe_synth.so")
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: run __graft_entry__.build()")
        L = C.CDLL(path)
        L.synth_gauss_f32.argtypes = [C.c_uint64, C.c_uint64, C.c_float, C.c_void_p, C.c_void_p]
        L.synth_gauss_f16.argtypes = [C.c_uint64, C.c_uint64, C.c_float, C.c_void_p, C.c_void_p]
        L.synth_affine.argtypes = [C.c_uint64, C.c_int, C.c_int, C.c_int, C.c_float,
                                   C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
        for f in (L.synth_gauss_f32, L.synth_gauss_f16, L.synth_affine):
            f.restype = C.c_int
        _gpu_lib = L
    return _gpu_lib


def _cur_stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def gpu_gauss(seed: int, tg: int, out, sigma: float):
    """Fill a CUDA tensor (float32, or float16/uint16 for fp16) like gauss()."""
    import torch
    n = out.numel()
    k = stream_key(seed, tg)
    sc = float(sigma_scale(sigma))
    if out.dtype == torch.float32:
        rc = _gpu().synth_gauss_f32(k, n, sc, out.data_ptr(), _cur_stream())
    else:
        assert out.element_size() == 2
        rc = _gpu().synth_gauss_f16(k, n, sc, out.data_ptr(), _cur_stream())
    if rc:
        raise RuntimeError(f"synth_gauss failed ({rc})")
    return out


def gpu_affine(seed: int, tg: int, rows: int, cols: int, bits: int, sigma: float, q, s, b):
    """Fill CUDA tensors q (int32/uint32 [rows][cols*bits/32]), s, b (16-bit
    [rows][cols/64]) like affine()."""
    rc = _gpu().synth_affine(stream_key(seed, tg), rows, cols, bits, float(sigma_scale(sigma)),
                             q.data_ptr(), s.data_ptr(), b.data_ptr(), _cur_stream())
    if rc:
        raise RuntimeError(f"synth_affine failed ({rc})")
