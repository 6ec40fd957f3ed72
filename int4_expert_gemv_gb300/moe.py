"""Thin Python binding of the C ABI in include/moe.h (ctypes).

Argument marshalling only: every function forwards device pointers, sizes and
the current CUDA stream to libmoe.so, which does all of the work.  Tensors are
PyTorch CUDA tensors (PyTorch supplies device memory and streams); raw integer
pointers are accepted wherever a tensor is.  A non-zero status raises
MoEError.  There is no fallback: if libmoe.so is missing the import of the
library fails loudly.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe.so")

MOE_OK, MOE_EINVAL, MOE_EUNSUPPORTED, MOE_ECUDA, MOE_ETIMEOUT, MOE_ENOSPACE = range(6)
MOE_DTYPE_F32, MOE_DTYPE_BF16 = 0, 1
MOE_PREC_AFFINE4, MOE_PREC_FP16 = 4, 16

_lock = threading.Lock()
_lib = None


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: {status_string(status)}: {detail}")
        self.status = status


# ------------------------------------------------------------------ structs
class HeadDesc(C.Structure):
    _fields_ = [("d", C.c_int), ("E", C.c_int), ("H", C.c_int), ("prec", C.c_int),
                ("fc1x", C.c_void_p), ("fc1_tab", C.c_void_p), ("b1", C.c_void_p),
                ("fc2", C.c_void_p), ("b2", C.c_void_p),
                ("lx", C.c_void_p), ("l_tab", C.c_void_p), ("bl", C.c_void_p)]


class LoraDesc(C.Structure):
    _fields_ = [("r", C.c_int), ("scale", C.c_float), ("A", C.c_void_p), ("B", C.c_void_p),
                ("a_stride", C.c_size_t), ("b_stride", C.c_size_t)]


class ExpertsDesc(C.Structure):
    _fields_ = [("d", C.c_int), ("F", C.c_int), ("E", C.c_int), ("bits", C.c_int),
                ("pool", C.c_void_p), ("expert_stride", C.c_size_t), ("shared", C.c_void_p),
                ("lora", LoraDesc * 3), ("shared_lora", LoraDesc * 3)]


class StackDesc(C.Structure):
    _fields_ = [("experts", C.c_void_p), ("routers", C.c_void_p), ("heads", C.c_void_p),
                ("n_layers", C.c_int), ("depth", C.c_int), ("K", C.c_int),
                ("self_predict", C.c_int), ("timeout_ns", C.c_ulonglong),
                ("debug_unset_wait", C.c_int), ("debug_trace", C.c_void_p),
                ("inflight_bytes", C.c_uint), ("slot_map", C.c_void_p),
                ("layer_ready", C.c_void_p), ("free_sms", C.c_int)]


class ChainInfo(C.Structure):
    _fields_ = [("smem_a", C.c_size_t), ("smem_b", C.c_size_t), ("threads", C.c_int),
                ("regs_a", C.c_int), ("regs_b", C.c_int),
                ("local_bytes_a", C.c_int), ("local_bytes_b", C.c_int),
                ("ctas_a", C.c_int), ("ctas_b", C.c_int), ("coresident", C.c_int)]


# ------------------------------------------------------------------ loading
def lib():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing: build it with "
                                  "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = C.CDLL(LIB_PATH)
            P, I, S = C.c_void_p, C.c_int, C.c_size_t
            sigs = {
                "moe_status_string": (C.c_char_p, [I]),
                "moe_last_error": (C.c_char_p, []),
                "moe_record_bytes": (S, [I, I]),
                "moe_packed_matrix_bytes": (S, [I, I, I]),
                "moe_pool_expert_bytes": (S, [I, I, I, I]),
                "moe_pack_matrix": (I, [P, P, P, I, I, I, P, P]),
                "moe_merge_lora": (I, [P, S, I, I, I, P, P, I, C.c_float, P, S, P]),
                "moe_gather_experts": (I, [P, S, I, P, I, S, P, S, P, P]),
                "moe_cache_experts": (I, [P, S, I, P, I, S, P, S, I, P, P, P, P, P, P, P]),
                "moe_pack_experts": (I, [I, I, I, I, P, P, P, P, P, P, P, P, P, P, S, P]),
                "moe_debug_dequant": (I, [P, I, I, I, I, P, P]),
                "moe_debug_batched_waits": (I, [C.c_ulonglong, I]),
                "moe_debug_batched_engine": (I, [I]),
                "moe_debug_batched_trace": (I, [P]),
                "moe_prerouter_head_workspace_bytes": (S, [C.POINTER(HeadDesc), I]),
                "moe_prerouter_head": (I, [C.POINTER(HeadDesc), P, I, P, P, I, I, P, P, S, P]),
                "moe_topk_route": (I, [P, I, I, I, P, P, P, P]),
                "moe_expert_ffn_workspace_bytes": (S, [C.POINTER(ExpertsDesc), I, I]),
                "moe_expert_ffn_int4": (I, [C.POINTER(ExpertsDesc), P, I, P, I, I, P, P, S, P]),
                "moe_combine_residual": (I, [P, P, I, I, I, I, P, P, P, P]),
                "moe_expert_ffn_int4_noalloc": (I, [C.POINTER(ExpertsDesc), P, I, P, I, I, P, P]),
                "moe_expert_ffn_noalloc_status": (I, [C.POINTER(C.c_int), P]),
                "moe_decode_step_workspace_bytes": (S, [C.POINTER(StackDesc)]),
                "moe_decode_step": (I, [C.POINTER(StackDesc), P, P, P, P, P, I, P, S, P]),
                "moe_decode_step_status": (I, [P, C.POINTER(C.c_int), P]),
                "moe_decode_step_chain_workspace_bytes": (S, [C.POINTER(StackDesc)]),
                "moe_decode_step_chain": (I, [C.POINTER(StackDesc), P, P, P, P, P, I, P, S, P]),
                "moe_decode_step_chain_info": (I, [C.POINTER(StackDesc), C.POINTER(ChainInfo)]),
                "moe_decode_step_chain_variant": (I, [I, I]),
                "moe_decode_step_chain_cache": (I, [I]),
            }
            for name, (res, args) in sigs.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def last_error() -> str:
    return lib().moe_last_error().decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoEError(rc, where, last_error())


def _nbytes(t):
    return 0 if t is None else (t.numel() * t.element_size() if not isinstance(t, int) else 0)


def _dtype_code(x) -> int:
    import torch
    if x.dtype == torch.float32:
        return MOE_DTYPE_F32
    if x.dtype == torch.bfloat16:
        return MOE_DTYPE_BF16
    raise TypeError(f"activations must be float32 or bfloat16, got {x.dtype}")


# ------------------------------------------------------------------ sizes
def moe_record_bytes(cols: int, bits: int) -> int:
    return lib().moe_record_bytes(cols, bits)


def moe_packed_matrix_bytes(rows: int, cols: int, bits: int) -> int:
    return lib().moe_packed_matrix_bytes(rows, cols, bits)


def moe_pool_expert_bytes(d: int, F: int, bits: int, group: int = 64) -> int:
    return lib().moe_pool_expert_bytes(d, F, bits, group)


def moe_prerouter_head_workspace_bytes(hd: HeadDesc, T: int) -> int:
    return lib().moe_prerouter_head_workspace_bytes(C.byref(hd), T)


def moe_expert_ffn_workspace_bytes(ed: ExpertsDesc, T: int, K: int) -> int:
    return lib().moe_expert_ffn_workspace_bytes(C.byref(ed), T, K)


# ------------------------------------------------------------------ calls
def moe_pack_matrix(q, s, b, rows: int, cols: int, bits: int, out, stream=None):
    _check(lib().moe_pack_matrix(_ptr(q), _ptr(s), _ptr(b), rows, cols, bits, _ptr(out),
                                 _stream(stream)), "moe_pack_matrix")


def moe_merge_lora(src, src_stride: int, rows: int, cols: int, bits: int, A, B, r: int,
                   scale: float, dst, dst_stride: int, stream=None):
    """W' = requantise(W + scale B A) on packed records (see include/moe.h).
    src / dst: tensors or device addresses (ints) of the first record."""
    _check(lib().moe_merge_lora(_ptr(src), src_stride, rows, cols, bits, _ptr(A), _ptr(B), r,
                                scale, _ptr(dst), dst_stride, _stream(stream)), "moe_merge_lora")


def moe_gather_experts(pool, expert_stride: int, E: int, idx, n: int, blob_bytes: int, slots,
                       slot_stride: int, slot_idx, stream=None):
    """Routed experts' blobs from a pool (HBM or pinned host memory) into HBM
    slots, route rewritten to the slots (see include/moe.h)."""
    _check(lib().moe_gather_experts(_ptr(pool), expert_stride, E, _ptr(idx), n, blob_bytes,
                                    _ptr(slots), slot_stride, _ptr(slot_idx), _stream(stream)),
           "moe_gather_experts")


def moe_cache_experts(pool, expert_stride: int, E: int, idx, n: int, blob_bytes: int, cache,
                      slot_stride: int, C: int, tags, ages, clock, slot_idx, plan, stats=None,
                      stream=None):
    """Route idx's experts through an HBM cache of C slots (LRU); slot_idx
    receives each entry's slot (the chain's slot map)."""
    _check(lib().moe_cache_experts(_ptr(pool), expert_stride, E, _ptr(idx), n, blob_bytes,
                                   _ptr(cache), slot_stride, C, _ptr(tags), _ptr(ages), _ptr(clock),
                                   _ptr(slot_idx), _ptr(plan), _ptr(stats), _stream(stream)),
           "moe_cache_experts")


def moe_pack_experts(d, F, E, bits, gate_q, gate_s, gate_b, up_q, up_s, up_b, down_q, down_s,
                     down_b, pool, expert_stride: int, stream=None):
    _check(lib().moe_pack_experts(d, F, E, bits, _ptr(gate_q), _ptr(gate_s), _ptr(gate_b),
                                  _ptr(up_q), _ptr(up_s), _ptr(up_b), _ptr(down_q),
                                  _ptr(down_s), _ptr(down_b), _ptr(pool), expert_stride,
                                  _stream(stream)), "moe_pack_experts")


def moe_debug_batched_waits(timeout_ns: int, stall: bool) -> None:
    """Test hook: the batched engine's wait bound (0 = 1 s) and a wait that
    nothing satisfies in every later launch (stall)."""
    _check(lib().moe_debug_batched_waits(int(timeout_ns), int(bool(stall))),
           "moe_debug_batched_waits")


def moe_debug_batched_engine(mode: int) -> None:
    """Which engine runs the batched GEMMs: 0 by size, 1 register
    (mma.sync), 2 tensor memory (tcgen05)."""
    _check(lib().moe_debug_batched_engine(int(mode)), "moe_debug_batched_engine")


def moe_debug_batched_trace(buf) -> None:
    """Profiling hook: stamps of CTA 0 of later tensor-memory engine launches
    into buf (device u64 [64 * 16]), or off (None)."""
    _check(lib().moe_debug_batched_trace(_ptr(buf)), "moe_debug_batched_trace")


def moe_debug_dequant(blob, d: int, F: int, bits: int, which: int, out, stream=None):
    _check(lib().moe_debug_dequant(_ptr(blob), d, F, bits, which, _ptr(out), _stream(stream)),
           "moe_debug_dequant")


def moe_prerouter_head(hd: HeadDesc, x, cur_idx, prev_idx, K: int, T: int, logits, ws,
                       stream=None, x_dtype: int | None = None):
    xd = _dtype_code(x) if x_dtype is None else x_dtype
    _check(lib().moe_prerouter_head(C.byref(hd), _ptr(x), xd, _ptr(cur_idx), _ptr(prev_idx), K,
                                    T, _ptr(logits), _ptr(ws), _nbytes(ws), _stream(stream)),
           "moe_prerouter_head")


def moe_topk_route(logits, T: int, E: int, K: int, idx, w, margin=None, stream=None):
    _check(lib().moe_topk_route(_ptr(logits), T, E, K, _ptr(idx), _ptr(w), _ptr(margin),
                                _stream(stream)), "moe_topk_route")


def moe_expert_ffn_int4(ed: ExpertsDesc, x, idx, T: int, K: int, y_slots, ws, stream=None,
                        x_dtype: int | None = None):
    xd = _dtype_code(x) if x_dtype is None else x_dtype
    _check(lib().moe_expert_ffn_int4(C.byref(ed), _ptr(x), xd, _ptr(idx), T, K, _ptr(y_slots),
                                     _ptr(ws), _nbytes(ws), _stream(stream)),
           "moe_expert_ffn_int4")


def moe_combine_residual(y_slots, w, T: int, K: int, has_shared: bool, d: int, residual, out,
                         x_next=None, stream=None):
    _check(lib().moe_combine_residual(_ptr(y_slots), _ptr(w), T, K, int(has_shared), d,
                                      _ptr(residual), _ptr(out), _ptr(x_next),
                                      _stream(stream)), "moe_combine_residual")


MOE_FFN_STATIC_SCRATCH_BYTES = 4 << 20


def moe_expert_ffn_int4_noalloc(ed: ExpertsDesc, x, idx, T: int, K: int, y_slots, stream=None,
                                x_dtype: int | None = None):
    """moe_expert_ffn_int4 for callers that cannot allocate: the library's
    fixed static device scratch stands in for the workspace."""
    xd = _dtype_code(x) if x_dtype is None else x_dtype
    _check(lib().moe_expert_ffn_int4_noalloc(C.byref(ed), _ptr(x), xd, _ptr(idx), T, K,
                                             _ptr(y_slots), _stream(stream)),
           "moe_expert_ffn_int4_noalloc")


def moe_expert_ffn_noalloc_status(stream=None) -> int:
    """Status word of the last allocation-free expert call on the current
    device (synchronises the stream): MOE_OK or MOE_ETIMEOUT."""
    st = C.c_int(0)
    _check(lib().moe_expert_ffn_noalloc_status(C.byref(st), _stream(stream)),
           "moe_expert_ffn_noalloc_status")
    return st.value


# ------------------------------------------------------------------ stack
def moe_decode_step_workspace_bytes(sd: StackDesc) -> int:
    return lib().moe_decode_step_workspace_bytes(C.byref(sd))


def moe_decode_step(sd: StackDesc, x0, out, route_idx, route_w, route_margin, t: int, ws,
                    stream=None):
    _check(lib().moe_decode_step(C.byref(sd), _ptr(x0), _ptr(out), _ptr(route_idx),
                                 _ptr(route_w), _ptr(route_margin), t, _ptr(ws), _nbytes(ws),
                                 _stream(stream)), "moe_decode_step")


def moe_decode_step_chain_workspace_bytes(sd: StackDesc) -> int:
    return lib().moe_decode_step_chain_workspace_bytes(C.byref(sd))


def moe_decode_step_chain(sd: StackDesc, x0, out, route_idx, route_w, route_margin, t: int, ws,
                          stream=None):
    _check(lib().moe_decode_step_chain(C.byref(sd), _ptr(x0), _ptr(out), _ptr(route_idx),
                                       _ptr(route_w), _ptr(route_margin), t, _ptr(ws), _nbytes(ws),
                                       _stream(stream)), "moe_decode_step_chain")


def moe_decode_step_chain_variant(variant: int, prefetch_l2: bool = True) -> None:
    """0: the library's choice, 1: two kernels per layer, 2: one cluster
    kernel per layer (process-wide; read when a step is enqueued)."""
    _check(lib().moe_decode_step_chain_variant(int(variant), int(bool(prefetch_l2))),
           "moe_decode_step_chain_variant")


def moe_decode_step_chain_cache(max_graphs: int) -> None:
    """Graphs moe_decode_step_chain keeps for repeated calls (0: none)."""
    _check(lib().moe_decode_step_chain_cache(int(max_graphs)), "moe_decode_step_chain_cache")


def moe_decode_step_chain_info(sd: StackDesc) -> dict:
    """How the chain's two per-layer kernels sit on an SM of the current
    device (shared memory, registers, CTAs per SM, co-residency)."""
    info = ChainInfo()
    _check(lib().moe_decode_step_chain_info(C.byref(sd), C.byref(info)),
           "moe_decode_step_chain_info")
    return {k: getattr(info, k) for k, _ in ChainInfo._fields_}


def moe_decode_step_status(ws, stream=None) -> int:
    st = C.c_int(0)
    _check(lib().moe_decode_step_status(_ptr(ws), C.byref(st), _stream(stream)),
           "moe_decode_step_status")
    return st.value
