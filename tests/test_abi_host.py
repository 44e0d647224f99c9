"""Host-side checks of the C ABI that need no GPU: the library loads,
exports every entry point the header declares, and rejects bad arguments
before it touches the device."""
import ctypes
import os
import re

import numpy as np
import pytest

import block_quantized_weight_02_gb300 as cq
from block_quantized_weight_02_gb300 import pack, synth
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    from block_quantized_weight_02_gb300 import build
    build.build()
    return cq.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "cq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cq_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ["cq_gemm_q4", "cq_gemm_q8row", "cq_moe_panels", "cq_moe_workspace_bytes", "cq_gemm_q4_workspace_bytes",
              "cq_dequant_q4", "cq_dequant_q8row", "cq_moe_layout", "cq_get_device_error", "cq_last_error"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in _declared():
        assert hasattr(L, n), n


def test_binding_names_match_the_abi(L):
    for n in _declared():
        assert hasattr(cq, n), n


FAKE = 0x10000   # 16-byte aligned, never dereferenced: validation fails first
ODD = 0x10008


def _q4(L, X=FAKE, xt=1, T=16, K=512, Wq=FAKE, Ws=FAKE, N=256, Y=FAKE, yt=2, ws=FAKE, wsb=1 << 30):
    return L.cq_gemm_q4(X, xt, T, K, Wq, Ws, N, Y, yt, ws, wsb, None)


def test_q4_validation(L):
    assert _q4(L, X=None) == 1
    assert _q4(L, Ws=None) == 1
    assert _q4(L, xt=2) == 2
    assert _q4(L, yt=0) == 2
    assert _q4(L, K=300) == 3
    assert _q4(L, K=128) == 3
    assert _q4(L, T=0) == 3
    assert _q4(L, N=0) == 3
    assert _q4(L, X=ODD) == 4
    assert _q4(L, Y=ODD) == 4
    assert _q4(L, wsb=10) == 6
    assert _q4(L, ws=FAKE + 16) == 6          # workspace must be 256-aligned
    assert "decline" in cq.cq_last_error()
    assert L.cq_last_launches() == 0          # a declined call launches nothing


def test_q8_validation(L):
    f = lambda **k: L.cq_gemm_q8row(k.get("X", FAKE), k.get("xt", 0), k.get("T", 4), k.get("K", 256),
                                    k.get("Wq", FAKE), k.get("rs", FAKE), k.get("N", 64), k.get("Y", FAKE),
                                    k.get("yt", 1), None)
    assert f(rs=None) == 1
    assert f(xt=5) == 2
    assert f(K=200) == 3
    assert f(Wq=ODD) == 4


def test_moe_validation(L):
    def f(**k):
        a = dict(X=FAKE, xt=1, T=32, H=2048, E=128, I=768, topk=8, idx=FAKE, w=FAKE, guq=FAKE, gus=FAKE, dq=FAKE,
                 ds=FAKE, Y=FAKE, yt=2, ws=FAKE, wsb=1 << 40)
        a.update(k)
        return L.cq_moe_panels(a["X"], a["xt"], a["T"], a["H"], a["E"], a["I"], a["topk"], a["idx"], a["w"],
                               a["guq"], a["gus"], a["dq"], a["ds"], a["Y"], a["yt"], a["ws"], a["wsb"], None)
    assert f(idx=None) == 1
    assert f(yt=0) == 2
    assert f(H=2000) == 3
    assert f(I=100) == 3
    assert f(topk=0) == 3
    assert f(E=2000) == 3
    assert f(w=ODD) == 4
    assert f(wsb=100) == 6


def test_workspace_sizes(L):
    # Q4: fp16 copy of X plus one f32 per row, each rounded up to 256 bytes
    assert cq.cq_gemm_q4_workspace_bytes(512, 4096) == 512 * 4096 * 2 + 2048
    assert cq.cq_gemm_q4_workspace_bytes(3, 256) == 1536 + 256
    b = cq.cq_moe_workspace_bytes(32, 2048, 768, 128, 8)
    P = 256
    # status, seg, perm, inv, active experts, 16 row-block counters, then the gathered rows and the panels' buffers
    need = 256 + 768 + P * 4 * 2 + 768 + 256 + P * 2048 * 2 + P * 4 + P * 768 * 4 + P * 768 * 2 + P * 4 + P * 2048 * 4
    assert b == need


def test_options(L):
    assert cq.lib().cq_set_option(99, 0) == 10
    assert cq.lib().cq_set_option(cq.CQ_OPT_SMALL_T_MAX, 33) == 10
    assert cq.lib().cq_set_option(cq.CQ_OPT_FORCE_PATH, 3) == 10
    assert cq.lib().cq_set_option(cq.CQ_OPT_WAIT_NS, 10) == 10
    old = cq.cq_get_option(cq.CQ_OPT_SMALL_T_MAX)
    cq.cq_set_option(cq.CQ_OPT_SMALL_T_MAX, 16)
    assert cq.cq_get_option(cq.CQ_OPT_SMALL_T_MAX) == 16
    cq.cq_set_option(cq.CQ_OPT_SMALL_T_MAX, old)
    # tcgen05 tiles, K split, operand placement and CTA pairs
    for opt, good, bad in [(cq.CQ_OPT_TC_BN, [0, 32, 64, 128, 192, 256], [16, 48, 512]),
                           (cq.CQ_OPT_TC_KSPLIT, [0, 1, 2], [3, -1]),
                           (cq.CQ_OPT_TC_AMODE, [0, 1, 2], [3]),
                           (cq.CQ_OPT_TC_PAIR, [0, 1, 2], [3, -1])]:
        before = cq.cq_get_option(opt)
        for v in good:
            assert cq.lib().cq_set_option(opt, v) == 0, (opt, v)
            assert cq.cq_get_option(opt) == v
        for v in bad:
            assert cq.lib().cq_set_option(opt, v) == 10, (opt, v)
        cq.cq_set_option(opt, before)


def test_packer_matches_oracle_packer():
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 16, (37, 512), dtype=np.uint8)
    assert np.array_equal(pack.pack_q4(codes), oracle.pack_q4(codes))
    assert np.array_equal(pack.unpack_q4_codes(pack.pack_q4(codes)), codes)
    stacked = rng.integers(0, 16, (3, 64, 256), dtype=np.uint8)
    ps = pack.pack_q4(stacked)
    for e in range(3):
        assert np.array_equal(ps[e], oracle.pack_q4(stacked[e]))


def test_widened_row_scales_exact():
    b = np.array([0x3C00, 0x0001, 0x7BFF, 0x211F], np.uint16)
    assert np.array_equal(pack.widen_f16_row_scales(b).astype(np.float64),
                          np.array([oracle.f16_to_f64(v) for v in b]))


def test_product_path_never_imports_oracle():
    """The library and binding stand alone: nothing in the package or the
    benchmark's GPU leg imports the oracle."""
    pkg = os.path.join(ROOT, "block_quantized_weight_02_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src and "oracle.c" not in src, f


def _ffn(L, X=FAKE, xt=1, T=16, H=512, I=768, g=FAKE, gs=FAKE, d=FAKE, ds=FAKE, Y=FAKE, yt=2, ws=FAKE, wsb=1 << 30):
    return L.cq_ffn_q4(X, xt, T, H, I, g, gs, d, ds, Y, yt, ws, wsb, None)


def test_ffn_validation(L):
    assert _ffn(L, X=None) == 1 and _ffn(L, ds=None) == 1 and _ffn(L, ws=None) == 1
    assert _ffn(L, xt=2) == 2 and _ffn(L, yt=0) == 2
    assert _ffn(L, T=0) == 3
    assert _ffn(L, H=384) == 3 and _ffn(L, I=128) == 3 and _ffn(L, I=300) == 3
    assert _ffn(L, g=ODD) == 4 and _ffn(L, Y=ODD) == 4
    need = L.cq_ffn_q4_workspace_bytes(16, 512, 768)
    # guarded X (16x512 fp16), its scales, a (16x768 f32), its fp16 copy and scales, each 256-aligned
    assert need == 16384 + 256 + 49152 + 24576 + 256
    assert _ffn(L, wsb=need - 1) == 6
    assert _ffn(L, ws=FAKE + 16) == 6
    assert "decline" in cq.cq_last_error()


def test_batched_validation(L):
    J = cq.cq_q4_job * 4
    good = J(*[cq.cq_q4_job(FAKE, FAKE, 0, 256 * j) for j in range(4)])
    call = lambda jobs=good, z=3, X=FAKE, T=16, K=512, ldx=512, N=256, Y=FAKE, ldy=1024, ws=FAKE, wsb=1 << 30: \
        L.cq_gemm_q4_batched(X, 1, T, K, ldx, ctypes.cast(jobs, ctypes.c_void_p), z, N, Y, 2, ldy, ws, wsb, None)
    assert call(X=None) == 1 and call(jobs=None) == 1
    assert call(z=0) == 10 and call(z=5) == 10
    assert call(K=384) == 3 and call(ldx=500) == 3 and call(ldy=700) == 3
    bad = J(cq.cq_q4_job(FAKE, FAKE, 4, 0), *[cq.cq_q4_job(FAKE, FAKE, 0, 0)] * 3)   # x_off not a multiple of 8
    assert call(jobs=bad, z=1) == 3
    bad = J(cq.cq_q4_job(FAKE, FAKE, 0, 900), *[cq.cq_q4_job(FAKE, FAKE, 0, 0)] * 3)  # y_off + N > ldy
    assert call(jobs=bad, z=1) == 3
    bad = J(cq.cq_q4_job(ODD, FAKE, 0, 0), *[cq.cq_q4_job(FAKE, FAKE, 0, 0)] * 3)
    assert call(jobs=bad, z=1) == 4
    assert L.cq_gemm_q4_batched_workspace_bytes(16, 512, 3) == 3 * (16 * 512 * 2 + 256)
    assert call(wsb=3 * (16 * 512 * 2 + 256) - 1) == 6


def test_route_validation(L):
    r = lambda T=4, E=16, k=4, sh=0, lg=FAKE, idx=FAKE, w=FAKE: L.cq_moe_route(lg, T, E, k, sh, idx, w, None)
    assert r(lg=None) == 1 and r(w=None) == 1
    assert r(T=0) == 3 and r(E=1025) == 3 and r(k=0) == 3 and r(k=17) == 3 and r(E=100, k=65) == 3 and r(sh=2) == 3
    assert r(lg=FAKE + 2) == 4


def test_format_variant_validation(L):
    q8b = lambda K=512, Ws=FAKE, ws=FAKE, wsb=1 << 30: L.cq_gemm_q8b(FAKE, 1, 16, K, FAKE, Ws, 64, FAKE, 2, ws, wsb, None)
    assert q8b(Ws=None) == 1 and q8b(K=192) == 3 and q8b(Ws=ODD) == 4 and q8b(wsb=100) == 6
    q4a = lambda K=512, gk=2, Wo=FAKE, wsb=1 << 30: L.cq_gemm_q4a(FAKE, 1, 16, K, FAKE, FAKE, Wo, gk, 64, FAKE, 2, FAKE,
                                                                  wsb, None)
    assert q4a(Wo=None) == 1 and q4a(gk=0) == 3 and q4a(gk=3) == 3 and q4a(K=384) == 3 and q4a(Wo=FAKE + 1) == 4
    assert q4a(K=65536, gk=1) == 3                                   # 2048 offsets per row > 512
    need = L.cq_gemm_q4a_workspace_bytes(16, 512, 64, 2)
    assert need == 16 * 512 * 2 + 256 + 16 * 8 * 4 + 16 * 64 * 4       # guard copy + scales, group sums, offset term
    assert q4a(wsb=need - 1) == 6
    q82 = lambda col=FAKE, K=512: L.cq_gemm_q8_2f(FAKE, 1, 16, K, FAKE, FAKE, col, 64, FAKE, 2, FAKE, 1 << 30, None)
    assert q82(col=None) == 1 and q82(K=200) == 3 and q82(col=ODD) == 4
