"""CPU oracle for the prerouted MoE decode layer (ctypes wrapper over oracle.c).

TEST INFRASTRUCTURE ONLY.  Imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; the product package never imports
it.  All arithmetic lives in ``oracle.c`` (plain C, fp64); this module only
builds the library with gcc and marshals numpy arrays.

Arrays handed in follow the logical storage formats of the synthetic inputs:
packed words ``q`` uint32 ``[rows][cols*bits/32]``, fp16 scale/bias bit
patterns ``s``/``b`` uint16 ``[rows][cols/64]``, fp16 matrices as uint16 bit
patterns.  Results come back as float64 numpy arrays.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

AFFINE, F16 = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc -O2, no fast-math, no FMA
    contraction: every operation rounds as written)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-Wall"]
    # OpenMP (row loops, see orc_set_threads) where the compiler has it
    r = subprocess.run(base + ["-fopenmp", "-o", tmp, _SRC, "-lm"], capture_output=True)
    if r.returncode != 0:
        subprocess.run(base + ["-Wno-unknown-pragmas", "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


# ---------------------------------------------------------------- structs
class Mat(C.Structure):
    _fields_ = [("kind", C.c_int), ("rows", C.c_int), ("cols", C.c_int),
                ("bits", C.c_int), ("group", C.c_int),
                ("q", C.c_void_p), ("s", C.c_void_p), ("b", C.c_void_p),
                ("f16", C.c_void_p)]


class Lora(C.Structure):
    _fields_ = [("r", C.c_int), ("scale", C.c_double),
                ("A", C.c_void_p), ("B", C.c_void_p)]


class Expert(C.Structure):
    _fields_ = [("gate", Mat), ("up", Mat), ("down", Mat),
                ("lg", Lora), ("lu", Lora), ("ld", Lora)]


class Head(C.Structure):
    _fields_ = [("d", C.c_int), ("E", C.c_int), ("H", C.c_int),
                ("fc1x", Mat), ("fc1_tab", C.c_void_p), ("b1", C.c_void_p),
                ("fc2", Mat), ("b2", C.c_void_p),
                ("lx", Mat), ("l_tab", C.c_void_p), ("bl", C.c_void_p)]


class Layer(C.Structure):
    _fields_ = [("experts", C.c_void_p), ("shared", C.c_void_p),
                ("router", Head), ("head", Head)]


class Stack(C.Structure):
    _fields_ = [("L", C.c_int), ("d", C.c_int), ("E", C.c_int), ("K", C.c_int),
                ("layers", C.c_void_p), ("single_layer_self_predict", C.c_int)]


class StackState(C.Structure):
    _fields_ = [("pred_idx", C.c_void_p), ("pred_z", C.c_void_p),
                ("pred_margin", C.c_void_p), ("prev_idx", C.c_void_p),
                ("t", C.c_int)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(_LIB_PATH)
            P = C.c_void_p
            L.orc_f16_to_f64.restype = C.c_double
            L.orc_f16_to_f64.argtypes = [C.c_uint16]
            L.orc_f64_to_f16.restype = C.c_uint16
            L.orc_f64_to_f16.argtypes = [C.c_double]
            L.orc_bf16_to_f64.restype = C.c_double
            L.orc_bf16_to_f64.argtypes = [C.c_uint16]
            L.orc_f64_to_bf16.restype = C.c_uint16
            L.orc_f64_to_bf16.argtypes = [C.c_double]
            L.orc_weight.restype = C.c_double
            L.orc_weight.argtypes = [C.POINTER(Mat), C.c_int, C.c_int]
            L.orc_dequant.argtypes = [C.POINTER(Mat), P]
            L.orc_gemv.argtypes = [C.POINTER(Mat), P, P]
            L.orc_set_threads.argtypes = [C.c_int]
            L.orc_set_threads.restype = None
            L.orc_openmp.argtypes = []
            L.orc_openmp.restype = C.c_int
            L.orc_lora_apply.argtypes = [C.POINTER(Lora), C.c_int, C.c_int, P, P]
            L.orc_silu.restype = C.c_double
            L.orc_silu.argtypes = [C.c_double]
            L.orc_gelu_erf.restype = C.c_double
            L.orc_gelu_erf.argtypes = [C.c_double]
            L.orc_expert_forward.argtypes = [C.POINTER(Expert), P, C.c_int, P, P]
            L.orc_expert_ffn.argtypes = [P, C.c_int, P, C.c_int, P, P, C.c_int,
                                         C.c_int, C.c_int, P]
            L.orc_head_features.argtypes = [C.c_int, C.c_int, P, P, P, C.c_int, P]
            L.orc_head_logits.argtypes = [C.POINTER(Head), P, P, P, C.c_int, P]
            L.orc_topk.argtypes = [P, C.c_int, C.c_int, P, P, P]
            L.orc_route_weights.argtypes = [P, P, C.c_int, P]
            L.orc_combine.argtypes = [P, P, C.c_int, C.c_int, C.c_int, P, P, P]
            L.orc_stack_step.argtypes = [C.POINTER(Stack), C.POINTER(StackState),
                                         P, P, C.c_double, P, P, P, P, P]
            L.orc_merge_weights.argtypes = [C.POINTER(Mat), C.POINTER(Lora), P]
            L.orc_quant_codes.argtypes = [P, C.c_int, C.c_int, C.c_int, C.c_int, P, P, P, P]
            L.orc_requantise.argtypes = [P, C.c_int, C.c_int, C.c_int, C.c_int, P, P, P, P, P, P]
            L.orc_merge_lora.argtypes = [C.POINTER(Mat), C.POINTER(Lora), P, P, P, P, P, P]
            _lib = L
    return _lib


# ---------------------------------------------------------------- helpers
def _p(a):
    return None if a is None else a.ctypes.data


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


class _Keep:
    """Holds numpy arrays alive for as long as a struct pointing at them."""

    def __init__(self):
        self.refs = []

    def add(self, a):
        if a is not None:
            a = np.ascontiguousarray(a)
            self.refs.append(a)
        return a


def mat(keep: _Keep, m: dict | None) -> Mat:
    """Struct for a weight matrix given as a dict.

    Affine: {"q": uint32 [rows][cols*bits/32], "s": uint16, "b": uint16,
    "rows", "cols", "bits", "group"}; fp16: {"f16": uint16 [rows][cols]}.
    """
    if m is None:
        return Mat()
    if "f16" in m:
        f = keep.add(np.asarray(m["f16"], dtype=np.uint16))
        return Mat(F16, f.shape[0], f.shape[1], 16, 0, None, None, None, _p(f))
    q = keep.add(np.asarray(m["q"], dtype=np.uint32))
    s = keep.add(np.asarray(m["s"], dtype=np.uint16))
    b = keep.add(np.asarray(m["b"], dtype=np.uint16))
    return Mat(AFFINE, m["rows"], m["cols"], m["bits"], m.get("group", 64),
               _p(q), _p(s), _p(b), None)


def lora(keep: _Keep, l: dict | None) -> Lora:
    if l is None:
        return Lora(0, 0.0, None, None)
    A = keep.add(np.asarray(l["A"], dtype=np.uint16))
    B = keep.add(np.asarray(l["B"], dtype=np.uint16))
    return Lora(A.shape[0], float(l["scale"]), _p(A), _p(B))


def expert(keep: _Keep, ex: dict) -> Expert:
    return Expert(mat(keep, ex["gate"]), mat(keep, ex["up"]), mat(keep, ex["down"]),
                  lora(keep, ex.get("lora_gate")), lora(keep, ex.get("lora_up")),
                  lora(keep, ex.get("lora_down")))


def head(keep: _Keep, hd: dict) -> Head:
    def opt(a):
        return None if a is None else _p(keep.add(np.asarray(a, dtype=np.uint16)))
    return Head(hd["d"], hd["E"], hd["H"],
                mat(keep, hd.get("fc1x")), opt(hd.get("fc1_tab")), opt(hd.get("b1")),
                mat(keep, hd.get("fc2")), opt(hd.get("b2")),
                mat(keep, hd["lx"]), opt(hd.get("l_tab")), opt(hd.get("bl")))


# ---------------------------------------------------------------- calls
def f16_to_f64(h: int) -> float:
    return lib().orc_f16_to_f64(h)


def f64_to_f16(v: float) -> int:
    return lib().orc_f64_to_f16(v)


def bf16_to_f64(h: int) -> float:
    return lib().orc_bf16_to_f64(h)


def f64_to_bf16(v: float) -> int:
    return lib().orc_f64_to_bf16(v)


def weight(m: dict, o: int, k: int) -> float:
    keep = _Keep()
    st = mat(keep, m)
    return lib().orc_weight(C.byref(st), o, k)


def dequant(m: dict) -> np.ndarray:
    keep = _Keep()
    st = mat(keep, m)
    w = np.zeros((st.rows, st.cols), np.float64)
    lib().orc_dequant(C.byref(st), _p(w))
    return w


def set_threads(n: int) -> None:
    """Threads for the oracle's row loops (results are identical at any
    count; 1 when the library was built without OpenMP)."""
    lib().orc_set_threads(int(n))


def openmp() -> bool:
    """Whether liboracle.so was built with OpenMP."""
    return bool(lib().orc_openmp())


def gemv(m: dict, x) -> np.ndarray:
    keep = _Keep()
    st = mat(keep, m)
    x = _f64(x)
    assert x.shape == (st.cols,)
    y = np.zeros(st.rows, np.float64)
    lib().orc_gemv(C.byref(st), _p(x), _p(y))
    return y


def merge_lora(m: dict, l: dict | None) -> dict:
    """W' = requantise(W + scale B A) group by group, in fp64 (oracle.h:
    orc_merge_lora); returns a matrix dict of m's shape plus the merged
    weights "w" [rows][cols] and the values before each rounding: "s_pre",
    "b_pre" [rows][cols/group], "t_pre" [rows][cols].  l None: W requantised."""
    keep = _Keep()
    st, sl = mat(keep, m), lora(keep, l)
    q = np.zeros((st.rows, st.cols * st.bits // 32), np.uint32)
    s = np.zeros((st.rows, st.cols // st.group), np.uint16)
    b = np.zeros_like(s)
    s_pre = np.zeros(s.shape, np.float64)
    b_pre = np.zeros(s.shape, np.float64)
    t_pre = np.zeros((st.rows, st.cols), np.float64)
    w = np.zeros((st.rows, st.cols), np.float64)
    lib().orc_merge_weights(C.byref(st), C.byref(sl), _p(w))
    lib().orc_requantise(_p(w), st.rows, st.cols, st.bits, st.group, _p(q), _p(s), _p(b),
                         _p(s_pre), _p(b_pre), _p(t_pre))
    return {"q": q, "s": s, "b": b, "rows": st.rows, "cols": st.cols, "bits": st.bits,
            "group": st.group, "w": w, "s_pre": s_pre, "b_pre": b_pre, "t_pre": t_pre}


def quant_codes(w, bits: int, group: int, s, b):
    """Codes of fp64 weights w [rows][cols] under given fp16 scales / biases
    (bit patterns [rows][cols/group]), and the values before rint (oracle.h:
    orc_quant_codes)."""
    w = np.ascontiguousarray(w, dtype=np.float64)
    rows, cols = w.shape
    s = np.ascontiguousarray(s, dtype=np.uint16)
    b = np.ascontiguousarray(b, dtype=np.uint16)
    q = np.zeros((rows, cols * bits // 32), np.uint32)
    t = np.zeros((rows, cols), np.float64)
    lib().orc_quant_codes(_p(w), rows, cols, bits, group, _p(s), _p(b), _p(q), _p(t))
    return q, t


def lora_apply(l: dict, x, y) -> np.ndarray:
    keep = _Keep()
    st = lora(keep, l)
    x = _f64(x)
    y = _f64(y).copy()
    lib().orc_lora_apply(C.byref(st), x.shape[0], y.shape[0], _p(x), _p(y))
    return y


def silu(g: float) -> float:
    return lib().orc_silu(g)


def gelu_erf(a: float) -> float:
    return lib().orc_gelu_erf(a)


def expert_forward(ex: dict, x, round_h_bf16: bool = False):
    keep = _Keep()
    st = expert(keep, ex)
    x = _f64(x)
    F, d = st.gate.rows, st.down.rows
    h = np.zeros(F, np.float64)
    y = np.zeros(d, np.float64)
    lib().orc_expert_forward(C.byref(st), _p(x), int(round_h_bf16), _p(h), _p(y))
    return h, y


def expert_ffn(experts: list, shared: dict | None, x, idx, round_h_bf16=False):
    """y_slots [T][K(+1)][d] for tokens x [T][d] routed to idx [T][K]."""
    keep = _Keep()
    arr = (Expert * len(experts))(*[expert(keep, e) for e in experts])
    sh = expert(keep, shared) if shared is not None else None
    x = _f64(x)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, K = idx.shape
    d = x.shape[1]
    slots = K + (shared is not None)
    y = np.zeros((T, slots, d), np.float64)
    lib().orc_expert_ffn(C.cast(arr, C.c_void_p), len(experts),
                         C.cast(C.pointer(sh), C.c_void_p) if sh is not None else None,
                         d, _p(x), _p(idx), T, K, int(round_h_bf16), _p(y))
    return y


def head_features(d, E, x, cur, prev, K):
    x = _f64(x)
    cur = None if cur is None else np.ascontiguousarray(cur, dtype=np.int32)
    prev = None if prev is None else np.ascontiguousarray(prev, dtype=np.int32)
    f = np.zeros(d + 2 * E, np.float64)
    lib().orc_head_features(d, E, _p(x), _p(cur), _p(prev), K, _p(f))
    return f


def head_logits(hd: dict, x, cur=None, prev=None, K: int = 0) -> np.ndarray:
    keep = _Keep()
    st = head(keep, hd)
    x = _f64(x)
    cur = None if cur is None else np.ascontiguousarray(cur, dtype=np.int32)
    prev = None if prev is None else np.ascontiguousarray(prev, dtype=np.int32)
    z = np.zeros(st.E, np.float64)
    lib().orc_head_logits(C.byref(st), _p(x), _p(cur), _p(prev), K, _p(z))
    return z


def topk(z, K: int):
    """(idx int32 [K], w float64 [K], margin float)."""
    z = _f64(z)
    idx = np.zeros(K, np.int32)
    w = np.zeros(K, np.float64)
    m = np.zeros(1, np.float64)
    lib().orc_topk(_p(z), z.shape[0], K, _p(idx), _p(w), _p(m))
    return idx, w, float(m[0])


def route_weights(z, idx) -> np.ndarray:
    z = _f64(z)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = np.zeros(idx.shape[0], np.float64)
    lib().orc_route_weights(_p(z), _p(idx), idx.shape[0], _p(w))
    return w


def combine(y_slots, w, has_shared: bool, residual, want_x_next: bool = True):
    y_slots = _f64(y_slots)
    w = _f64(w)
    residual = _f64(residual)
    K = w.shape[0]
    d = residual.shape[0]
    out = np.zeros(d, np.float64)
    xn = np.zeros(d, np.float64) if want_x_next else None
    lib().orc_combine(_p(y_slots), _p(w), K, int(has_shared), d, _p(residual),
                      _p(out), _p(xn))
    return out, xn


class StackRunner:
    """Holds an oracle stack (structs + arrays) and its route state."""

    def __init__(self, layers: list, d: int, E: int, K: int,
                 single_layer_self_predict: bool = False):
        self.keep = _Keep()
        self.L, self.d, self.E, self.K = len(layers), d, E, K
        self._experts = []
        lay = []
        for ly in layers:
            arr = (Expert * len(ly["experts"]))(*[expert(self.keep, e) for e in ly["experts"]])
            self._experts.append(arr)
            sh = None
            if ly.get("shared") is not None:
                sh = C.pointer(expert(self.keep, ly["shared"]))
                self._experts.append(sh)
            hd = head(self.keep, ly["head"]) if ly.get("head") is not None else Head()
            lay.append(Layer(C.cast(arr, C.c_void_p),
                             C.cast(sh, C.c_void_p) if sh is not None else None,
                             head(self.keep, ly["router"]), hd))
        self.layers = (Layer * len(lay))(*lay)
        self.stack = Stack(self.L, d, E, K, C.cast(self.layers, C.c_void_p),
                           int(single_layer_self_predict))
        self.pred_idx = np.zeros((self.L, K), np.int32)
        self.pred_z = np.zeros((self.L, E), np.float64)
        self.pred_margin = np.zeros(self.L, np.float64)
        self.prev_idx = np.zeros((self.L, K), np.int32)
        self.state = StackState(_p(self.pred_idx), _p(self.pred_z),
                                _p(self.pred_margin), _p(self.prev_idx), 0)

    def step(self, x0, ext_idx=None, tie_margin: float = 1e-4):
        x0 = _f64(x0)
        ext = None if ext_idx is None else np.ascontiguousarray(ext_idx, dtype=np.int32)
        out = np.zeros(self.d, np.float64)
        used_idx = np.zeros((self.L, self.K), np.int32)
        used_w = np.zeros((self.L, self.K), np.float64)
        used_margin = np.zeros(self.L, np.float64)
        forced = np.zeros(self.L, np.uint8)
        lib().orc_stack_step(C.byref(self.stack), C.byref(self.state), _p(x0),
                             _p(ext), tie_margin, _p(out), _p(used_idx),
                             _p(used_w), _p(used_margin), _p(forced))
        return dict(out=out, idx=used_idx, w=used_w, margin=used_margin,
                    forced=forced.astype(bool))
