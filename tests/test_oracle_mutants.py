"""Plausible mistakes planted in a copy of the oracle must fail the pins.

Each mutant is a text edit of oracle.c compiled into a temporary library;
the hand-built blocks and the addressing pin are then run against it.
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

from test_oracle import _golden_blocks

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "oracle.c")

MUTANTS = {
    "nibbles_swapped": ("(int)(byte & 15) - 8) * d;\n                w[n * K + 32 * b + 16 + i] = (float)((int)(byte >> 4)",
                        "(int)(byte >> 4) - 8) * d;\n                w[n * K + 32 * b + 16 + i] = (float)((int)(byte & 15)"),
    "offset_7": ("(float)((int)(byte & 15) - 8)", "(float)((int)(byte & 15) - 7)"),
    "scale_index_drops_row": ("ws[n * (K / 32) + b]", "ws[b]"),
    "interleaved_elements": ("w[n * K + 32 * b + 16 + i]", "w[n * K + 32 * b + 2 * (i % 8) + 1 + 16 * (i / 8)]"),
    "subnormal_flush": ("v = ldexp((double)f, -24);", "v = 0.0;"),
}


def _build_mutant(name, tmp):
    src = open(SRC).read()
    old, new = MUTANTS[name]
    assert old in src, name
    path = os.path.join(tmp, f"{name}.c")
    open(path, "w").write(src.replace(old, new, 1))
    so = os.path.join(tmp, f"{name}.so")
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", path, "-o", so, "-lm"])
    return ctypes.CDLL(so)


def _dequant(lib, wq, ws, N, K):
    out = np.empty((N, K), np.float32)
    lib.or_dequant_q4(ctypes.c_void_p(wq.ctypes.data), ctypes.c_void_p(ws.ctypes.data),
                      ctypes.c_int64(N), ctypes.c_int64(K), ctypes.c_void_p(out.ctypes.data))
    return out


def _pins_pass(lib):
    for name, sbits, sval, raw, m in _golden_blocks():
        wq = np.frombuffer(raw, np.uint8).reshape(1, 16).copy()
        ws = np.array([[sbits]], np.uint16)
        got = _dequant(lib, wq, ws, 1, 32)[0]
        exp = np.array([mi * sval for mi in m], np.float64).astype(np.float32)
        if not np.array_equal(got.view(np.uint32), exp.view(np.uint32)):
            return False
    # two rows x two blocks with distinct scales (the addressing pin)
    blocks = {b[0]: b for b in _golden_blocks()}
    grid = [["ramp_one", "pos03"], ["ramp_ncent", "pos20"]]
    wq = np.zeros((2, 32), np.uint8)
    ws = np.zeros((2, 2), np.uint16)
    exp = np.zeros((2, 64), np.float32)
    for n in range(2):
        for b in range(2):
            _, sb, sv, raw, m = blocks[grid[n][b]]
            wq[n, 16 * b:16 * b + 16] = np.frombuffer(raw, np.uint8)
            ws[n, b] = sb
            exp[n, 32 * b:32 * b + 32] = np.array([mi * sv for mi in m], np.float32)
    return np.array_equal(_dequant(lib, wq, ws, 2, 64).view(np.uint32), exp.view(np.uint32))


def test_unmutated_copy_passes():
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "orig.c")
        open(path, "w").write(open(SRC).read())
        so = os.path.join(tmp, "orig.so")
        subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", path, "-o", so, "-lm"])
        assert _pins_pass(ctypes.CDLL(so))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_pins(name):
    with tempfile.TemporaryDirectory() as tmp:
        assert not _pins_pass(_build_mutant(name, tmp)), f"mutant {name} slipped through"


# ---- the dense FFN chain: mutants against its one-hot closed form ----------

FFN_MUTANTS = {
    "ffn_gate_up_swapped": ("g += (double)wgu[i * H + k] * x[k];\n                for (int64_t k = 0; k < H; k++) u += (double)wgu[(I + i) * H + k] * x[k];",
                            "u += (double)wgu[i * H + k] * x[k];\n                for (int64_t k = 0; k < H; k++) g += (double)wgu[(I + i) * H + k] * x[k];"),
    "ffn_silu_sign": ("                a[i] = g / (1.0 + exp(-g)) * u;\n                if (A_out)",
                      "                a[i] = g / (1.0 + exp(g)) * u;\n                if (A_out)"),
    "ffn_down_transposed": ("wd[n * I + i]", "wd[i * H + n]"),
    "ffn_down_skips_last": ("for (int64_t i = 0; i < I; i++) {\n                    double p", "for (int64_t i = 0; i + 1 < I; i++) {\n                    double p"),
}


def _ffn_closed_form_passes(lib):
    import math
    H = I = 64
    rng = np.random.default_rng(71)
    gc = rng.integers(0, 16, (2 * I, H), dtype=np.uint8)
    dc = rng.integers(0, 16, (H, I), dtype=np.uint8)
    pack = lambda c: (c.reshape(c.shape[0], -1, 2, 16)[:, :, 0, :] | (c.reshape(c.shape[0], -1, 2, 16)[:, :, 1, :] << 4)).reshape(c.shape[0], -1).astype(np.uint8)
    guq, dq = pack(gc), pack(dc)
    gus = np.full((2 * I, H // 32), 0x3C00, np.uint16)
    ds = np.full((H, I // 32), 0x3C00, np.uint16)
    ks = [5, 30]
    X = np.zeros((2, H))
    X[[0, 1], ks] = 1.0
    Y = np.empty((2, H))
    S = np.empty((2, H))
    p = lambda a: ctypes.c_void_p(a.ctypes.data)
    i64 = ctypes.c_int64
    lib.or_ffn(p(X), i64(2), i64(H), i64(I), p(guq), p(gus), p(dq), p(ds), p(Y), p(S), None)
    wd = dc.astype(np.float64) - 8
    for t, k in enumerate(ks):
        a = [(g - 8) / (1 + math.exp(-(g - 8))) * (u - 8) for g, u in zip(gc[:I, k].astype(float), gc[I:, k].astype(float))]
        y = np.array([math.fsum(wd[n] * a) for n in range(H)])
        if not np.allclose(Y[t], y, rtol=1e-12, atol=1e-12):
            return False
    return True


def test_unmutated_ffn_passes():
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "orig.c")
        open(path, "w").write(open(SRC).read())
        so = os.path.join(tmp, "orig.so")
        subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", path, "-o", so, "-lm"])
        assert _ffn_closed_form_passes(ctypes.CDLL(so))


@pytest.mark.parametrize("name", sorted(FFN_MUTANTS))
def test_ffn_mutant_fails_closed_form(name):
    src = open(SRC).read()
    old, new = FFN_MUTANTS[name]
    assert src.count(old) == 1, name
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, f"{name}.c")
        open(path, "w").write(src.replace(old, new))
        so = os.path.join(tmp, f"{name}.so")
        subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", path, "-o", so, "-lm"])
        assert not _ffn_closed_form_passes(ctypes.CDLL(so)), f"mutant {name} slipped through"


# ---- routing: mutants against the library argsort and the closed-form weights ----

ROUTE_MUTANTS = {
    "route_ties_prefer_higher_index": ("(best < 0 || l[e] > l[best])", "(best < 0 || l[e] >= l[best])"),
    "route_no_renormalise": ("w[t * slots + j] = (float)(p[j] / wsum);", "w[t * slots + j] = (float)p[j];"),
    "route_shared_sign": ("(1.0 / (1.0 + exp(-(double)l[E])))", "(1.0 / (1.0 + exp((double)l[E])))"),
}


def _route_pins_pass(lib):
    rng = np.random.default_rng(83)
    lg = np.ascontiguousarray(np.concatenate([rng.integers(-2, 3, (20, 16)).astype(np.float32) * 0.5,
                                              np.full((20, 1), np.log(3.0), np.float32)], axis=1))
    T, E, k = 20, 16, 4
    idx = np.empty((T, k + 1), np.int32)
    w = np.empty((T, k + 1), np.float32)
    p = lambda a: ctypes.c_void_p(a.ctypes.data)
    lib.or_route(p(lg), ctypes.c_int64(T), ctypes.c_int64(E), ctypes.c_int64(k), ctypes.c_int(1), p(idx), p(w))
    if not np.array_equal(idx[:, :k], np.argsort(-lg[:, :E], axis=1, kind="stable")[:, :k]):
        return False
    if not np.allclose(w[:, :k].sum(axis=1), 1.0, rtol=1e-6):
        return False
    return bool(np.all(np.abs(w[:, k] - 0.75) < 1e-7))


@pytest.mark.parametrize("name", sorted(ROUTE_MUTANTS) + ["none"])
def test_route_mutants_fail_pins(name):
    src = open(SRC).read()
    if name != "none":
        old, new = ROUTE_MUTANTS[name]
        assert src.count(old) == 1, name
        src = src.replace(old, new)
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, f"{name}.c")
        open(path, "w").write(src)
        so = os.path.join(tmp, f"{name}.so")
        subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", path, "-o", so, "-lm"])
        assert _route_pins_pass(ctypes.CDLL(so)) == (name == "none")


# ---- format variants: mutants against their pins ----------------------------

FORMAT_MUTANTS = {
    "q8b_scale_per_16": ("s[n * (K / 32) + k / 32]", "s[n * (K / 32) + k / 16 % (K / 32)]"),
    "q4a_offset_per_block": ("off[n * gpr + (k / 32) / gk]", "off[n * gpr + (k / 32) % gpr]"),
    "q8_2f_col_by_row": ("(double)col[k] * X[t * K + k]", "(double)col[n % K] * X[t * K + k]"),
}


def _format_pins_pass(lib):
    p = lambda a: ctypes.c_void_p(a.ctypes.data)
    i64 = ctypes.c_int64
    rng = np.random.default_rng(97)
    # Q8 per 32: one f32 rounding of q * s[n][k/32]
    q = rng.integers(-128, 128, (4, 128)).astype(np.int8)
    s = rng.uniform(1e-3, 1e-2, (4, 4)).astype(np.float32)
    w = np.empty((4, 128), np.float32)
    lib.or_dequant_q8b(p(q), p(s), i64(4), i64(128), p(w))
    if not np.array_equal(w, (q.astype(np.float64) * np.repeat(s.astype(np.float64), 32, axis=1)).astype(np.float32)):
        return False
    # affine Q4, gk = 2: (nibble - 8) * 1 + offset of the group
    codes = rng.integers(0, 16, (3, 256)).astype(np.uint8)
    wq = (codes.reshape(3, -1, 2, 16)[:, :, 0, :] | (codes.reshape(3, -1, 2, 16)[:, :, 1, :] << 4)).reshape(3, -1).astype(np.uint8)
    ws = np.full((3, 8), 0x3C00, np.uint16)
    offv = rng.integers(-8, 8, (3, 4)).astype(np.float32) * 0.125
    off = np.ascontiguousarray((offv.view(np.uint32) >> 16).astype(np.uint16))
    w = np.empty((3, 256), np.float32)
    lib.or_dequant_q4a(p(wq), p(ws), p(off), i64(2), i64(3), i64(256), p(w))
    if not np.array_equal(w, (codes.astype(np.float32) - 8) + np.repeat(offv, 64, axis=1)):
        return False
    # q8_2f: unit activations pick one column: Y = rs * q[n][k] * col[k]
    q = rng.integers(-128, 128, (6, 64)).astype(np.int8)
    rs = np.full(6, 0.5, np.float32)
    col = rng.integers(1, 8, 64).astype(np.float32)
    X = np.zeros((2, 64))
    X[0, 5] = X[1, 40] = 1.0
    Y = np.empty((2, 6))
    S = np.empty((2, 6))
    lib.or_gemm_q8_2f(p(q), p(rs), p(col), p(X), i64(2), i64(6), i64(64), p(Y), p(S))
    return np.array_equal(Y[0], 0.5 * q[:, 5] * col[5]) and np.array_equal(Y[1], 0.5 * q[:, 40] * col[40])


@pytest.mark.parametrize("name", sorted(FORMAT_MUTANTS) + ["none"])
def test_format_mutants_fail_pins(name):
    src = open(SRC).read()
    if name != "none":
        old, new = FORMAT_MUTANTS[name]
        assert src.count(old) == 1, name
        src = src.replace(old, new)
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, f"{name}.c")
        open(path, "w").write(src)
        so = os.path.join(tmp, f"{name}.so")
        subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", path, "-o", so, "-lm"])
        assert _format_pins_pass(ctypes.CDLL(so)) == (name == "none")
