"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, sizes its buffers correctly and rejects bad arguments before it
enqueues anything (these calls never reach the device)."""
import ctypes as C
import os
import re

import pytest

from int4_expert_gemv_gb300 import build as nbuild
from int4_expert_gemv_gb300.configs import ALL, MOE35B, TINY

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def m():
    nbuild.build()
    from int4_expert_gemv_gb300 import moe
    moe.lib()
    return moe


def _declared(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(m):
    names = _declared("moe.h")
    assert "moe_expert_ffn_int4" in names and "moe_prerouter_head" in names
    assert len(names) >= 14
    lib = C.CDLL(m.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(m):
    assert m.status_string(0) == "MOE_OK"
    assert m.status_string(1) == "MOE_EINVAL"
    assert m.status_string(4) == "MOE_ETIMEOUT"
    assert m.status_string(99) == "MOE_UNKNOWN"


def test_pool_expert_bytes_matches_the_page(m):
    vals = {}
    for line in open(os.path.join(GOLDEN, "page_values.txt")):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split("=")
            vals[k.strip()] = float(v)
    n = m.moe_pool_expert_bytes(int(vals["expert_bytes.d_model"]), int(vals["expert_bytes.ffn"]),
                                int(vals["expert_bytes.bits"]), int(vals["expert_bytes.group"]))
    assert n == 7_077_888 == vals["expert_bytes.value_mib"] * 2 ** 20


def test_sizes(m):
    assert m.moe_record_bytes(2048, 4) == 1024 + 128
    assert m.moe_record_bytes(512, 4) == 256 + 32
    assert m.moe_record_bytes(128, 4) == 80           # 64 + 8, padded to 16
    assert m.moe_record_bytes(4096, 2) == 1024 + 256
    assert m.moe_record_bytes(100, 4) == 0 and m.moe_record_bytes(128, 3) == 0
    assert m.moe_pool_expert_bytes(2048, 512, 4, 64) == MOE35B.expert_bytes()
    assert m.moe_pool_expert_bytes(4096, 1024, 2, 64) == ALL["wide-int2"].expert_bytes()
    assert m.moe_pool_expert_bytes(256, 128, 4, 64) >= TINY.expert_bytes()
    assert m.moe_pool_expert_bytes(256, 128, 4, 32) == 0
    assert m.moe_packed_matrix_bytes(3, 2048, 4) == 3 * 1152


def _experts_desc(m, **kw):
    ed = m.ExpertsDesc()
    ed.d, ed.F, ed.E, ed.bits = 2048, 512, 256, 4
    ed.pool = 1 << 20
    ed.expert_stride = m.moe_pool_expert_bytes(2048, 512, 4, 64)
    for k, v in kw.items():
        setattr(ed, k, v)
    return ed


def _ffn(m, ed, T=1, K=4, x=1 << 20, idx=1 << 20, y=1 << 20, ws=1 << 20, ws_bytes=1 << 30,
         x_dtype=0):
    return m.lib().moe_expert_ffn_int4(C.byref(ed), x, x_dtype, idx, T, K, y, ws, ws_bytes, None)


@pytest.mark.parametrize("kw,call", [
    (dict(d=2000), {}), (dict(F=500), {}), (dict(bits=3), {}), (dict(E=0), {}),
    (dict(pool=None), {}), (dict(pool=(1 << 20) + 16), {}), (dict(expert_stride=1024), {}),
    ({}, dict(K=0)), ({}, dict(K=17)), ({}, dict(T=-1)), ({}, dict(x=None)),
    ({}, dict(x=(1 << 20) + 4)), ({}, dict(idx=None)), ({}, dict(x_dtype=7)),
])
def test_expert_ffn_rejects_bad_arguments(m, kw, call):
    assert _ffn(m, _experts_desc(m, **kw), **call) == m.MOE_EINVAL
    assert m.last_error() != ""


@pytest.mark.parametrize("kw,call", [
    (dict(d=2000), {}), (dict(E=0), {}), (dict(E=-5), {}),
    (dict(pool=None), {}), ({}, dict(K=0)), ({}, dict(K=17)), ({}, dict(K=40)),
    ({}, dict(T=-1)), ({}, dict(x=None)), ({}, dict(x=(1 << 20) + 4)), ({}, dict(x_dtype=7)),
    ({}, dict(T=100000, x=(1 << 20) + 4)),
])
def test_noalloc_rejects_bad_arguments_like_the_workspace_entry(m, kw, call):
    """The allocation-free entry validates before it sizes its scratch: bad
    arguments get MOE_EINVAL (as from moe_expert_ffn_int4), never
    MOE_ENOSPACE, and touch no device."""
    ed = _experts_desc(m, **kw)
    a = dict(T=1, K=4, x=1 << 20, idx=1 << 20, y=1 << 20, x_dtype=0)
    a.update(call)
    rc = m.lib().moe_expert_ffn_int4_noalloc(C.byref(ed), a["x"], a["x_dtype"], a["idx"],
                                              a["T"], a["K"], a["y"], None)
    assert rc == m.MOE_EINVAL, m.last_error()


def test_expert_ffn_rejects_small_workspace(m):
    ed = _experts_desc(m)
    need = m.moe_expert_ffn_workspace_bytes(ed, 1, 4)
    assert need > 0
    assert _ffn(m, ed, ws_bytes=need - 1) == m.MOE_ENOSPACE
    assert _ffn(m, ed, ws=None) == m.MOE_ENOSPACE


def test_expert_ffn_rejects_bad_lora(m):
    ed = _experts_desc(m)
    ed.lora[2] = m.LoraDesc(65, 1.0, 1 << 20, 1 << 20, 0, 0)
    assert _ffn(m, ed) == m.MOE_EINVAL
    ed.lora[2] = m.LoraDesc(8, 1.0, None, 1 << 20, 0, 0)
    assert _ffn(m, ed) == m.MOE_EINVAL


def test_empty_batch_is_a_no_op(m):
    # T == 0 returns before touching any pointer or the device
    assert _ffn(m, _experts_desc(m), T=0, x=None, idx=None, y=None, ws=None) == m.MOE_OK
    assert m.lib().moe_topk_route(None, 0, 256, 4, None, None, None, None) == m.MOE_OK
    assert m.lib().moe_combine_residual(None, None, 0, 4, 1, 2048, None, None, None, None) == m.MOE_OK


def _head_desc(m, **kw):
    hd = m.HeadDesc()
    hd.d, hd.E, hd.H, hd.prec = 2048, 256, 512, m.MOE_PREC_AFFINE4
    hd.fc1x = hd.fc2 = hd.lx = 1 << 20
    for k, v in kw.items():
        setattr(hd, k, v)
    return hd


@pytest.mark.parametrize("kw", [dict(d=100), dict(E=0), dict(E=2000), dict(H=100),
                                dict(prec=8), dict(lx=None), dict(fc1x=None), dict(fc2=None)])
def test_head_rejects_bad_descriptors(m, kw):
    hd = _head_desc(m, **kw)
    rc = m.lib().moe_prerouter_head(C.byref(hd), 1 << 20, 0, None, None, 4, 1, 1 << 20,
                                    1 << 20, 1 << 30, None)
    assert rc == m.MOE_EINVAL


def test_head_workspace_and_k_checks(m):
    hd = _head_desc(m)
    need = m.moe_prerouter_head_workspace_bytes(hd, 3)
    # status word (256 bytes), g [T][H] fp32, zl [T][E] fp32, sums of x per group
    # [T][ld] fp32 (ld = d/64 padded to 4), g split into bf16 hi/lo rows
    # [2T][H], their sums per group [2T][ldh], each 256-aligned
    a256 = lambda n: (n + 255) // 256 * 256
    ld = (hd.d // 64 + 3) // 4 * 4
    ldh = (hd.H // 64 + 3) // 4 * 4
    assert need == (256 + a256(3 * 512 * 4) + a256(3 * 256 * 4) + a256(3 * ld * 4)
                    + a256(6 * 512 * 2) + a256(6 * ldh * 4))
    rc = m.lib().moe_prerouter_head(C.byref(hd), 1 << 20, 0, None, None, 4, 3, 1 << 20,
                                    1 << 20, need - 1, None)
    assert rc == m.MOE_ENOSPACE
    rc = m.lib().moe_prerouter_head(C.byref(hd), 1 << 20, 0, 1 << 20, None, 0, 3, 1 << 20,
                                    1 << 20, need, None)
    assert rc == m.MOE_EINVAL


@pytest.mark.parametrize("T,E,K", [(1, 0, 1), (1, 2000, 4), (1, 256, 0), (1, 256, 17), (1, 4, 5)])
def test_topk_rejects_bad_shapes(m, T, E, K):
    assert m.lib().moe_topk_route(1 << 20, T, E, K, 1 << 20, 1 << 20, None, None) == m.MOE_EINVAL


def test_combine_rejects_bad_arguments(m):
    L = m.lib()
    assert L.moe_combine_residual(1 << 20, 1 << 20, 1, 4, 1, 0, 1 << 20, 1 << 20, None, None) == m.MOE_EINVAL
    assert L.moe_combine_residual(1 << 20, None, 1, 4, 1, 64, 1 << 20, 1 << 20, None, None) == m.MOE_EINVAL
    assert L.moe_combine_residual(1 << 20, None, 1, 0, 0, 64, 1 << 20, 1 << 20, None, None) == m.MOE_EINVAL


def test_pack_rejects_bad_arguments(m):
    L = m.lib()
    assert L.moe_pack_matrix(1 << 20, 1 << 20, 1 << 20, 4, 100, 4, 1 << 20, None) == m.MOE_EINVAL
    assert L.moe_pack_matrix(1 << 20, 1 << 20, 1 << 20, 4, 128, 4, (1 << 20) + 16, None) == m.MOE_EINVAL
    assert L.moe_pack_experts(2048, 512, 4, 4, *([1 << 20] * 9), 1 << 20, 4096, None) == m.MOE_EINVAL
    assert L.moe_debug_dequant(1 << 20, 2048, 512, 4, 3, 1 << 20, None) == m.MOE_EINVAL


def _stack(m, shared_ranks, depth=1):
    """A one-layer decode stack descriptor with placeholder device pointers
    (validation runs before any pointer is used)."""
    eds = (m.ExpertsDesc * 1)()
    ed = eds[0]
    ed.d, ed.F, ed.E, ed.bits = 2048, 512, 256, 4
    ed.pool, ed.shared = 1 << 20, 1 << 21
    ed.expert_stride = m.moe_pool_expert_bytes(2048, 512, 4, 64)
    for j, r in enumerate(shared_ranks):
        ed.shared_lora[j] = m.LoraDesc(r, 1.0, 1 << 20, 1 << 20, 0, 0) if r else m.LoraDesc()
    rts = (m.HeadDesc * 1)()
    rts[0].d, rts[0].E, rts[0].prec, rts[0].lx = 2048, 256, m.MOE_PREC_AFFINE4, 1 << 20
    sd = m.StackDesc()
    sd.experts, sd.routers = C.addressof(eds), C.addressof(rts)
    sd.n_layers, sd.depth, sd.K = 1, depth, 4
    return sd, (eds, rts)


@pytest.mark.parametrize("entry", ["moe_decode_step", "moe_decode_step_chain"])
def test_decode_step_rejects_wide_shared_gate_up_lora(m, entry):
    """The shared expert's gate and up adapters share one 32-wide A x vector:
    ranks 20 + 20 are refused before anything is enqueued; 16 + 16 gets past
    the descriptor checks (to the NULL-pointer check that follows)."""
    p = 1 << 20
    for ranks, want in (((20, 20, 0), m.MOE_EUNSUPPORTED), ((16, 16, 0), m.MOE_EINVAL)):
        sd, keep = _stack(m, ranks)
        rc = getattr(m.lib(), entry)(C.byref(sd), p, None, p, p, p, 1, p, 1 << 30, None)
        assert rc == want, (ranks, m.last_error())
    assert "NULL" in m.last_error()


def test_merge_lora_rejects_bad_arguments(m):
    L = m.lib()
    p = 1 << 20
    rb = m.moe_record_bytes(512, 4)
    ok = dict(src=p, ss=rb, rows=4, cols=512, bits=4, A=p, B=p, r=8, scale=2.0, dst=p, ds=rb)

    def call(**kw):
        a = dict(ok, **kw)
        return L.moe_merge_lora(a["src"], a["ss"], a["rows"], a["cols"], a["bits"], a["A"], a["B"],
                                a["r"], a["scale"], a["dst"], a["ds"], None)
    for bad in (dict(bits=3), dict(cols=500), dict(rows=-1), dict(r=-1), dict(A=None),
                dict(B=None), dict(src=None), dict(dst=None), dict(ss=rb - 16), dict(ds=rb + 4),
                dict(src=p + 4)):
        assert call(**bad) == m.MOE_EINVAL, bad
        assert m.last_error() != ""
    assert call(rows=0, src=None, dst=None) == m.MOE_OK      # nothing to do, nothing touched


def test_gather_experts_rejects_bad_arguments(m):
    L = m.lib()
    p = 1 << 20
    ok = dict(pool=p, st=4096, E=8, idx=p, n=4, blob=4096, slots=p, ss=4096, sidx=p)

    def call(**kw):
        a = dict(ok, **kw)
        return L.moe_gather_experts(a["pool"], a["st"], a["E"], a["idx"], a["n"], a["blob"],
                                    a["slots"], a["ss"], a["sidx"], None)
    for bad in (dict(n=-1), dict(n=18), dict(E=0), dict(pool=None), dict(idx=None),
                dict(slots=None), dict(sidx=None), dict(blob=0), dict(blob=4008),
                dict(st=2048), dict(ss=4100), dict(pool=p + 8)):
        assert call(**bad) == m.MOE_EINVAL, bad
    assert call(n=0, pool=None) == m.MOE_OK


def test_expert_sections_match_the_blob_layout(m):
    """Gate row f = record 2f, up row f = record 2f + 1 of the gate/up
    section; the down section on the next 256-byte boundary; the blob size
    covers both (the layout the header states)."""
    from int4_expert_gemv_gb300.model import expert_sections
    for cfg in (MOE35B, TINY, ALL["wide-int2"]):
        (g_off, g_st, g_rows, g_cols), (u_off, u_st, u_rows, u_cols), (d_off, d_st, d_rows, d_cols) = \
            expert_sections(cfg)
        rec_d, rec_f = m.moe_record_bytes(cfg.d, cfg.bits), m.moe_record_bytes(cfg.F, cfg.bits)
        assert (g_off, g_st, g_rows, g_cols) == (0, 2 * rec_d, cfg.F, cfg.d)
        assert (u_off, u_st, u_rows, u_cols) == (rec_d, 2 * rec_d, cfg.F, cfg.d)
        assert d_off % 256 == 0 and 2 * cfg.F * rec_d <= d_off < 2 * cfg.F * rec_d + 256
        assert (d_st, d_rows, d_cols) == (rec_f, cfg.d, cfg.F)
        assert d_off + cfg.d * rec_f <= m.moe_pool_expert_bytes(cfg.d, cfg.F, cfg.bits, 64)


def test_decode_step_chain_validation(m):
    """The chained entry checks its arguments before touching the device:
    step 0 (every layer routes itself) is refused, NULL buffers and a short
    or unaligned workspace are refused, and a 2-bit stack whose d is not a
    multiple of 256 is unsupported."""
    L = m.lib()
    p = 1 << 20
    sd, keep = _stack(m, (16, 16, 16))
    need = L.moe_decode_step_chain_workspace_bytes(C.byref(sd))
    assert need > 0
    call = lambda **kw: L.moe_decode_step_chain(
        C.byref(kw.get("sd", sd)), kw.get("x0", p), kw.get("out", p), p, p, p, kw.get("t", 1),
        kw.get("ws", p), kw.get("nb", need), None)
    assert call(t=0) == m.MOE_EINVAL
    assert call(x0=None) == m.MOE_EINVAL and call(out=None) == m.MOE_EINVAL
    assert call(nb=need - 1) == m.MOE_ENOSPACE
    assert call(ws=p + 16) == m.MOE_ENOSPACE
    sd2, keep2 = _stack(m, (0, 0, 0))
    e = C.cast(sd2.experts, C.POINTER(m.ExpertsDesc))[0]
    e.d, e.bits = 320, 2
    e.expert_stride = m.moe_pool_expert_bytes(320, 512, 2, 64)
    r = C.cast(sd2.routers, C.POINTER(m.HeadDesc))[0]
    r.d = 320
    need2 = L.moe_decode_step_chain_workspace_bytes(C.byref(sd2))
    assert need2 > 0
    assert L.moe_decode_step_chain(C.byref(sd2), p, p, p, p, p, 1, p, need2, None) == m.MOE_EUNSUPPORTED


def test_chain_variant_and_cache_settings(m):
    """The decode-chain settings validate their arguments on the host: an
    unknown variant or a cache size outside 0 .. 1024 is MOE_EINVAL; valid
    values are accepted (and put back to the defaults)."""
    lib = m.lib()
    assert lib.moe_decode_step_chain_variant(3, 1) == m.MOE_EINVAL
    assert lib.moe_decode_step_chain_variant(-1, 1) == m.MOE_EINVAL
    assert lib.moe_decode_step_chain_cache(-1) == m.MOE_EINVAL
    assert lib.moe_decode_step_chain_cache(1025) == m.MOE_EINVAL
    for v in (1, 2, 0):
        assert lib.moe_decode_step_chain_variant(v, 1) == m.MOE_OK
    assert lib.moe_decode_step_chain_cache(0) == m.MOE_OK
    assert lib.moe_decode_step_chain_cache(16) == m.MOE_OK
