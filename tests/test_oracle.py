"""Pins of the CPU oracle against facts fixed outside it.

Each test checks an oracle function against something it does not share
code with: hand-built blocks (tests/golden), a second statement of the
format on the same page (GGUF Q4_0), numpy/torch conversions and matmuls,
exact rational arithmetic, closed forms and invariants.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from block_quantized_weight_02_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_blocks():
    out = []
    for line in open(os.path.join(GOLDEN, "q4_blocks.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, sbits, sval, bytes_, m = [f.strip() for f in line.split(";")]
        out.append((name, int(sbits, 16), float(sval), bytes.fromhex(bytes_.replace(" ", "")),
                    [float(v) for v in m.split()]))
    return out


def _bits32(a):
    return np.asarray(a, np.float32).view(np.uint32)


# ---- number formats --------------------------------------------------------

def test_f16_decode_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(b) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint64), ref[~nan].view(np.uint64))


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_to_f64(b) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_x_to_f64_both_types():
    rng = np.random.default_rng(11)
    v = rng.standard_normal(1000)
    h = v.astype(np.float16)
    assert np.array_equal(oracle.x_to_f64(h.view(np.uint16), "f16"), h.astype(np.float64))
    b = synth.f32_to_bf16_bits(v.astype(np.float32))
    ref = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(oracle.x_to_f64(b, "bf16"), ref)


# Hand-derived single roundings of f64 to bf16 (8 significant bits, ties to
# even, subnormal quantum 2^-133, overflow past the largest finite value).
BF16_CASES = [
    (1.0, 0x3F80),
    (-1.0, 0xBF80),
    (-0.0, 0x8000),
    (1 + 2**-8, 0x3F80),                # tie -> even (down)
    (1 + 3 * 2**-8, 0x3F82),            # tie -> even (up)
    (1 + 2**-8 + 2**-30, 0x3F81),       # just above the tie
    (1 + 2**-8 + 2**-25, 0x3F81),       # an f32 intermediate would round to the tie, then down
    (2.0**-133, 0x0001),                # smallest subnormal
    (2.0**-134, 0x0000),                # half of it: tie -> even (zero)
    (3 * 2.0**-135, 0x0001),            # 0.75 quantum -> 1 quantum
    ((2 - 2**-7) * 2.0**127, 0x7F7F),   # largest finite
    ((2 - 2**-8) * 2.0**127, 0x7F80),   # tie at the top -> even = overflow
    (float("inf"), 0x7F80),
    (-float("inf"), 0xFF80),
]


@pytest.mark.parametrize("x,bits", BF16_CASES)
def test_f64_to_bf16_hand_cases(x, bits):
    assert int(oracle.f64_to_bf16(np.array([x]))[0]) == bits


def _bf16_exact_rne(fr: Fraction) -> Fraction:
    """Nearest multiple of the bf16 quantum at |fr|, ties to even (exact)."""
    if fr == 0:
        return Fraction(0)
    a = abs(fr)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** max(e - 7, -133)
    n = a / q
    lo = math.floor(n)
    rem = n - lo
    r = lo + 1 if (rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1)) else lo
    v = r * q
    return v if fr > 0 else -v


def test_f64_to_bf16_random_vs_exact_fractions():
    rng = np.random.default_rng(5)
    v = np.concatenate([rng.standard_normal(400) * 10.0 ** rng.integers(-30, 30, 400),
                        1 + rng.integers(0, 1 << 20, 100) * 2.0**-20])
    got = oracle.f64_to_bf16(v)
    for x, g in zip(v, got):
        ref = _bf16_exact_rne(Fraction(float(x)))
        assert Fraction(oracle.bf16_to_f64(int(g))) == ref


def test_f64_to_f32_is_numpy_cast():
    rng = np.random.default_rng(6)
    v = rng.standard_normal(1000) * 1e3
    assert np.array_equal(oracle.f64_to_f32(v), v.astype(np.float32))


# ---- Q4 dequantization -----------------------------------------------------

@pytest.mark.parametrize("blk", _golden_blocks(), ids=lambda b: b[0])
def test_dequant_q4_golden_block(blk):
    name, sbits, sval, raw, m = blk
    assert float(np.uint16(sbits).view(np.float16)) == sval or (sval == 0.0)
    wq = np.frombuffer(raw, np.uint8).reshape(1, 16)
    ws = np.array([[sbits]], np.uint16)
    got = oracle.dequant_q4(wq, ws, 1, 32)[0]
    exp = np.array([mi * sval for mi in m], np.float64).astype(np.float32)
    assert np.array_equal(_bits32(got), _bits32(exp)), name  # bit-exact, zero signs included


def test_dequant_q4_row_and_block_addressing():
    """Blocks land at n*K/2 + 16b with the scale at n*(K/32) + b."""
    blocks = {b[0]: b for b in _golden_blocks()}
    grid = [["ramp_one", "pos03"], ["ramp_ncent", "pos20"]]     # [row][block]
    wq = np.zeros((2, 32), np.uint8)
    ws = np.zeros((2, 2), np.uint16)
    exp = np.zeros((2, 64), np.float32)
    for n in range(2):
        for b in range(2):
            _, sbits, sval, raw, m = blocks[grid[n][b]]
            wq[n, 16 * b:16 * b + 16] = np.frombuffer(raw, np.uint8)
            ws[n, b] = sbits
            exp[n, 32 * b:32 * b + 32] = np.array([mi * sval for mi in m], np.float32)
    got = oracle.dequant_q4(wq, ws, 2, 64)
    assert np.array_equal(_bits32(got), _bits32(exp))


def _q4_0_decode_block(block18: bytes) -> np.ndarray:
    """The GGUF Q4_0 decoder on the same page, read for what it states: an
    fp16 d, then 16 bytes; the 4-wide output group i holds (low nibble - 8)
    * d of bytes 4i..4i+3 and group i+4 the high nibbles of the same bytes."""
    d = float(np.frombuffer(block18[:2], np.float16)[0])
    q = block18[2:]
    out = np.zeros(32, np.float32)
    for i in range(4):
        for c in range(4):
            v = q[4 * i + c]
            out[4 * i + c] = np.float32(((v & 15) - 8)) * np.float32(d)
            out[4 * (i + 4) + c] = np.float32(((v >> 4) - 8)) * np.float32(d)
    return out


def test_dequant_q4_matches_gguf_q4_0_statement():
    rng = np.random.default_rng(9)
    N, K = 6, 128
    wq = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    ws = rng.uniform(-2, 2, (N, K // 32)).astype(np.float16).view(np.uint16)
    got = oracle.dequant_q4(wq, ws, N, K)
    for n in range(N):
        for b in range(K // 32):
            blk = ws[n, b].tobytes() + wq[n, 16 * b:16 * b + 16].tobytes()
            assert np.array_equal(got[n, 32 * b:32 * b + 32], _q4_0_decode_block(blk))


def test_pack_q4_inverts_to_codes():
    """pack then dequant with scale 1.0 gives codes - 8 in element order."""
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 16, (5, 96), dtype=np.uint8)
    wq = oracle.pack_q4(codes)
    ws = np.full((5, 3), 0x3C00, np.uint16)
    assert np.array_equal(oracle.dequant_q4(wq, ws, 5, 96), codes.astype(np.float32) - 8)
    # byte 16b+i: low nibble = element 32b+i, high = element 32b+16+i
    assert wq[2, 16 + 5] == (codes[2, 32 + 5] | (codes[2, 32 + 21] << 4))


# ---- Q8-row ----------------------------------------------------------------

def test_dequant_q8row_is_one_f32_product():
    rng = np.random.default_rng(4)
    q, rs = synth.draw_q8row(rng, 7, 64)
    got = oracle.dequant_q8row(q, rs)
    exp = (q.astype(np.float64) * rs.astype(np.float64)[:, None]).astype(np.float32)
    assert np.array_equal(got, exp)
    q2 = np.array([[-128, 127, 0, -1]], np.int8)
    assert np.array_equal(oracle.dequant_q8row(q2, np.array([0.5], np.float32)),
                          np.array([[-64.0, 63.5, 0.0, -0.5]], np.float32))


# ---- GEMM ------------------------------------------------------------------

def _exact_dequant(wq, ws, N, K):
    """Fractions from the hand-checked block rule (independent of the C code)."""
    out = [[None] * K for _ in range(N)]
    for n in range(N):
        for b in range(K // 32):
            d = Fraction(float(np.uint16(ws[n, b]).view(np.float16)))
            for i in range(16):
                byte = int(wq[n, 16 * b + i])
                out[n][32 * b + i] = ((byte & 15) - 8) * d
                out[n][32 * b + 16 + i] = ((byte >> 4) - 8) * d
    return out


@pytest.mark.parametrize("T,N,K", [(1, 1, 32), (2, 2, 64), (3, 5, 32), (3, 5, 64)])
def test_gemm_q4_vs_exact_rationals(T, N, K):
    case = synth.gemm_q4_case(100 + T * N + K, T, K, N, x_dtype="bf16", signed=True)
    wq = oracle.pack_q4(case["codes"])
    X = oracle.x_to_f64(case["x"], "bf16")
    Y, S = oracle.gemm_q4(wq, case["scales"], N, K, X)
    W = _exact_dequant(wq, case["scales"], N, K)
    for t in range(T):
        for n in range(N):
            exact = sum(W[n][k] * Fraction(float(X[t, k])) for k in range(K))
            sabs = sum(abs(W[n][k] * Fraction(float(X[t, k]))) for k in range(K))
            # recursive f64 summation: |err| <= (K-1) u sum|p|, u = 2^-53
            assert abs(Fraction(Y[t, n]) - exact) <= Fraction(K, 2**53) * sabs
            assert Fraction(S[t, n]) == sabs or abs(Fraction(S[t, n]) - sabs) <= Fraction(K, 2**53) * sabs
            # final roundings agree with rounding the exact value (away from ties)
            ef = float(exact)
            assert abs(float(np.float32(Y[t, n])) - ef) <= abs(ef) * 2**-23 + 1e-300
            assert Fraction(oracle.bf16_to_f64(int(oracle.f64_to_bf16(np.array([Y[t, n]]))[0]))) \
                in (_bf16_exact_rne(exact), _bf16_exact_rne(Fraction(Y[t, n])))


def test_gemm_matches_torch_f64_matmul():
    case = synth.gemm_q4_case(21, 37, 512, 192, x_dtype="bf16")
    wq = oracle.pack_q4(case["codes"])
    W = oracle.dequant_q4(wq, case["scales"], 192, 512)
    X = oracle.x_to_f64(case["x"], "bf16")
    Y, S = oracle.gemm(W, X)
    ref = (torch.from_numpy(X) @ torch.from_numpy(W.astype(np.float64)).T).numpy()
    assert np.all(np.abs(Y - ref) <= 512 * 2.0**-52 * S)
    assert np.allclose(S, np.abs(X) @ np.abs(W.astype(np.float64)).T, rtol=1e-12)


def test_gemm_sampled_equals_full():
    case = synth.gemm_q4_case(22, 9, 256, 40)
    wq = oracle.pack_q4(case["codes"])
    X = oracle.x_to_f64(case["x"], "bf16")
    Y, S = oracle.gemm_q4(wq, case["scales"], 40, 256, X)
    tn = np.array([[0, 0], [8, 39], [3, 17], [5, 5]], np.int64)
    ys, ss = oracle.gemm_q4_sampled(wq, case["scales"], 40, 256, X, tn)
    assert np.array_equal(ys, Y[tn[:, 0], tn[:, 1]]) and np.array_equal(ss, S[tn[:, 0], tn[:, 1]])
    q8 = synth.gemm_q8_case(23, 9, 256, 40)
    X8 = oracle.x_to_f64(q8["x"], "bf16")
    Y8, S8 = oracle.gemm_q8row(q8["q"], q8["rs"], X8)
    ys8, ss8 = oracle.gemm_q8_sampled(q8["q"], q8["rs"], X8, tn)
    assert np.array_equal(ys8, Y8[tn[:, 0], tn[:, 1]]) and np.array_equal(ss8, S8[tn[:, 0], tn[:, 1]])


def test_gemm_doubling_scales_doubles_y_exactly():
    case = synth.gemm_q4_case(24, 5, 256, 33)
    wq = oracle.pack_q4(case["codes"])
    X = oracle.x_to_f64(case["x"], "bf16")
    Y1, _ = oracle.gemm_q4(wq, case["scales"], 33, 256, X)
    s2 = (case["scales"].view(np.float16).astype(np.float32) * 2).astype(np.float16).view(np.uint16)
    Y2, _ = oracle.gemm_q4(wq, s2, 33, 256, X)
    assert np.array_equal(Y2, 2 * Y1)


def test_q8row_with_unit_scale_equals_q4_with_unit_scales():
    case = synth.gemm_q4_case(25, 4, 128, 16)
    wq = oracle.pack_q4(case["codes"])
    X = oracle.x_to_f64(case["x"], "bf16")
    ones = np.full((16, 4), 0x3C00, np.uint16)
    Yq4, Sq4 = oracle.gemm_q4(wq, ones, 16, 128, X)
    q8 = case["codes"].astype(np.int16) - 8
    Yq8, Sq8 = oracle.gemm_q8row(q8.astype(np.int8), np.ones(16, np.float32), X)
    assert np.array_equal(Yq4, Yq8) and np.array_equal(Sq4, Sq8)


def test_q8row_scale_on_result_vs_scaled_weights():
    """Row scale on the f64 sum vs on each weight: equal within f32 rounding."""
    case = synth.gemm_q8_case(26, 6, 256, 20)
    X = oracle.x_to_f64(case["x"], "bf16")
    Ya, S = oracle.gemm_q8row(case["q"], case["rs"], X)
    Yb, _ = oracle.gemm(oracle.dequant_q8row(case["q"], case["rs"]), X)
    assert np.all(np.abs(Ya - Yb) <= 2.0**-24 * S + 1e-300)


# ---- MoE -------------------------------------------------------------------

def test_moe_layout_is_stable_sort_by_expert():
    rng = np.random.default_rng(12)
    T, topk, E = 75, 3, 8
    idx = rng.integers(0, E, (T, topk)).astype(np.int32)
    idx[idx == 5] = 6                     # expert 5 unused
    perm, seg = oracle.moe_layout(idx, E)
    ref = np.argsort(idx.reshape(-1), kind="stable")
    assert np.array_equal(perm, ref)
    counts = np.bincount(idx.reshape(-1), minlength=E)
    assert np.array_equal(seg, np.concatenate([[0], np.cumsum(counts)]))
    assert seg[5] == seg[6]


def test_moe_layout_rejects_out_of_range():
    with pytest.raises(ValueError):
        oracle.moe_layout(np.array([[0, 4]], np.int32), 4)
    with pytest.raises(ValueError):
        oracle.moe_layout(np.array([[0, -1]], np.int32), 4)


def _one_hot_expert(H, I, k, gate_codes, up_codes, seed):
    """An expert whose gate row i and up row i hold gate_codes[i] / up_codes[i]
    at column k (nibble 8 = 0 elsewhere), scales 1.0; a random down matrix."""
    gcodes = np.full((2 * I, H), 8, np.uint8)
    gcodes[:I, k] = gate_codes
    gcodes[I:, k] = up_codes
    rng = np.random.default_rng(seed)
    dcodes = rng.integers(0, 16, (H, I), dtype=np.uint8)
    dsc = rng.uniform(0.005, 0.02, (H, I // 32)).astype(np.float16).view(np.uint16)
    return (oracle.pack_q4(gcodes), np.full((2 * I, H // 32), 0x3C00, np.uint16),
            oracle.pack_q4(dcodes), dsc, dcodes)


def test_moe_pair_closed_form_one_hot_input():
    """x = unit vector e_k: g_i = gate[i][k], u_i = up[i][k] exactly, so the
    chain reduces to a = silu(g) * u and o = Wd . a."""
    H, I, k = 64, 32, 37
    rng = np.random.default_rng(31)
    gc = rng.integers(0, 16, I).astype(np.uint8)
    uc = rng.integers(0, 16, I).astype(np.uint8)
    guq, gus, dq, ds, dcodes = _one_hot_expert(H, I, k, gc, uc, 32)
    x = np.zeros(H)
    x[k] = 1.0
    a, o, s = oracle.moe_pair(oracle.dequant_q4(guq, gus, 2 * I, H), oracle.dequant_q4(dq, ds, H, I), x)
    g = gc.astype(np.float64) - 8
    u = uc.astype(np.float64) - 8
    a_ref = np.array([gi / (1 + math.exp(-gi)) * ui for gi, ui in zip(g, u)])
    assert np.allclose(a, a_ref, rtol=1e-15, atol=0)
    wd = (dcodes.astype(np.float64) - 8) * ds.view(np.float16).astype(np.float64).repeat(32, axis=1)
    o_ref = np.array([math.fsum(wd[n] * a_ref) for n in range(H)])
    assert np.allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(s, np.abs(wd) @ np.abs(a_ref), rtol=1e-12)


def _small_moe(seed, T=6, H=64, I=32, E=5, topk=2):
    c = synth.moe_case(seed, T=T, H=H, I=I, E=E, topk=topk)
    guq = np.stack([oracle.pack_q4(c["gu_codes"][e]) for e in range(E)])
    dq = np.stack([oracle.pack_q4(c["d_codes"][e]) for e in range(E)])
    return c, guq, dq


def test_moe_all_slots_one_expert_equals_dense_chain():
    c, guq, dq = _small_moe(41)
    T, H, I, E = c["T"], c["H"], c["I"], c["E"]
    idx = np.full((T, 4), 3, np.int32)
    w = np.tile(np.array([0.5, 0.25, 0.125, 0.125], np.float32), (T, 1))
    X = oracle.x_to_f64(c["x"], "bf16")
    Y, _ = oracle.moe(X, idx, w, guq, c["gu_scales"], dq, c["d_scales"], E, I)
    wgu = oracle.dequant_q4(guq[3], c["gu_scales"][3], 2 * I, H)
    wd = oracle.dequant_q4(dq[3], c["d_scales"][3], H, I)
    for t in range(T):
        _, o, _ = oracle.moe_pair(wgu, wd, X[t])
        assert np.allclose(Y[t], o, rtol=1e-14, atol=1e-14)


def test_moe_unrouted_expert_contributes_nothing_and_slot_order_is_free():
    c, guq, dq = _small_moe(42)
    E, I = c["E"], c["I"]
    X = oracle.x_to_f64(c["x"], "bf16")
    idx = np.array([[0, 1], [1, 2], [2, 0], [0, 2], [1, 0], [2, 1]], np.int32)   # experts 3, 4 unused
    w = np.array([[0.6, 0.4]] * 6, np.float32)
    Y, S = oracle.moe(X, idx, w, guq, c["gu_scales"], dq, c["d_scales"], E, I)
    # scrambling the unused experts' weights changes nothing
    gs2 = c["gu_scales"].copy()
    gs2[3:] = 0x3C00
    Y2, _ = oracle.moe(X, idx, w, guq, gs2, dq, c["d_scales"], E, I)
    assert np.array_equal(Y, Y2)
    # swapping each row's two slots (with their weights) leaves Y unchanged up to rounding
    Y3, _ = oracle.moe(X, idx[:, ::-1].copy(), w[:, ::-1].copy(), guq, c["gu_scales"], dq, c["d_scales"], E, I)
    assert np.all(np.abs(Y3 - Y) <= 4 * 2.0**-52 * S)


def test_moe_weight_linearity_and_gate_up_order():
    """Y is linear in the routing weights, and swapping the gate and up
    halves of an expert changes the result (silu(g) u != silu(u) g)."""
    c, guq, dq = _small_moe(43, T=3)
    E, I, H = c["E"], c["I"], c["H"]
    X = oracle.x_to_f64(c["x"], "bf16")
    idx = np.array([[4], [4], [4]], np.int32)
    Y1, _ = oracle.moe(X, idx, np.ones((3, 1), np.float32), guq, c["gu_scales"], dq, c["d_scales"], E, I)
    Yh, _ = oracle.moe(X, idx, np.full((3, 1), 0.5, np.float32), guq, c["gu_scales"], dq, c["d_scales"], E, I)
    assert np.array_equal(Yh, 0.5 * Y1)
    guq_sw = guq.copy()
    gus_sw = c["gu_scales"].copy()
    guq_sw[4] = np.concatenate([guq[4][I:], guq[4][:I]])
    gus_sw[4] = np.concatenate([c["gu_scales"][4][I:], c["gu_scales"][4][:I]])
    Ysw, _ = oracle.moe(X, idx, np.ones((3, 1), np.float32), guq_sw, gus_sw, dq, c["d_scales"], E, I)
    assert not np.allclose(Ysw, Y1)


def test_moe_rejects_out_of_range_index():
    c, guq, dq = _small_moe(44, T=2)
    X = oracle.x_to_f64(c["x"], "bf16")
    with pytest.raises(ValueError):
        oracle.moe(X, np.array([[0, 5], [1, 2]], np.int32), np.ones((2, 2), np.float32),
                   guq, c["gu_scales"], dq, c["d_scales"], c["E"], c["I"])


# ---- routing (the input recipe) ---------------------------------------------

def test_routing_ties_prefer_lower_index_and_renormalise():
    logits = np.array([[0.5, 2.0, 2.0, -1.0, 2.0, 0.5]], np.float32)
    idx, w = synth.route_topk(logits, 4)
    assert idx.tolist() == [[1, 2, 4, 0]]
    assert abs(float(w.sum()) - 1.0) < 1e-6
    p = np.exp(np.array([2.0, 2.0, 2.0, 0.5]) - 2.0)
    assert np.allclose(w[0], p / p.sum(), rtol=1e-6)


# ---- dense FFN chain -------------------------------------------------------

def _dense_ffn_weights(seed, H, I):
    rng = np.random.default_rng(seed)
    gc, gs = synth.draw_q4(rng, 2 * I, H, signed=True)
    dc, ds = synth.draw_q4(rng, H, I, signed=True)
    return oracle.pack_q4(gc), gs, oracle.pack_q4(dc), ds


def test_ffn_closed_form_one_hot_rows():
    """Token t = unit vector e_{k_t}: g_i = gate[i][k_t], u_i = up[i][k_t]
    exactly, a_i = silu(g_i) u_i, then y = Wd . a; a and y written out with
    math.exp and exact sums (fsum)."""
    H, I = 64, 32
    rng = np.random.default_rng(61)
    gc = np.full((2 * I, H), 8, np.uint8)
    gc[:, :] = rng.integers(0, 16, (2 * I, H))
    guq = oracle.pack_q4(gc)
    gus = np.full((2 * I, H // 32), 0x3C00, np.uint16)          # scale 1: weights are nibble - 8
    dc = rng.integers(0, 16, (H, I), dtype=np.uint8)
    ds = rng.uniform(0.005, 0.02, (H, I // 32)).astype(np.float16).view(np.uint16)
    dq = oracle.pack_q4(dc)
    ks = [3, 17, 40, 63]
    X = np.zeros((len(ks), H))
    X[np.arange(len(ks)), ks] = 1.0
    Y, S, A = oracle.ffn(X, guq, gus, dq, ds, I, want_a=True)
    wd = (dc.astype(np.float64) - 8) * ds.view(np.float16).astype(np.float64).repeat(32, axis=1)
    for t, k in enumerate(ks):
        g = gc[:I, k].astype(np.float64) - 8
        u = gc[I:, k].astype(np.float64) - 8
        a = np.array([gi / (1 + math.exp(-gi)) * ui for gi, ui in zip(g, u)])
        assert np.allclose(A[t], a, rtol=1e-15, atol=0)
        y = np.array([math.fsum(wd[n] * a) for n in range(H)])
        assert np.allclose(Y[t], y, rtol=1e-12, atol=1e-12)
        assert np.allclose(S[t], np.abs(wd) @ np.abs(a), rtol=1e-12)


def test_ffn_equals_one_expert_moe_with_unit_weight():
    """The dense chain is the routed chain with one expert and weight 1 for
    every token: equal to oracle.moe (E=1, top-1) bit for bit, and each row
    equal to moe_pair on that token."""
    H, I, T = 128, 64, 5
    guq, gus, dq, ds = _dense_ffn_weights(62, H, I)
    rng = np.random.default_rng(63)
    X = oracle.x_to_f64(synth.draw_x(rng, T, H), "bf16")
    Y, S = oracle.ffn(X, guq, gus, dq, ds, I)
    Ym, Sm = oracle.moe(X, np.zeros((T, 1), np.int32), np.ones((T, 1), np.float32), guq[None], gus[None],
                        dq[None], ds[None], 1, I)
    assert np.array_equal(Y, Ym) and np.array_equal(S, Sm)
    wgu = oracle.dequant_q4(guq, gus, 2 * I, H)
    wd = oracle.dequant_q4(dq, ds, H, I)
    for t in range(T):
        _, o, s = oracle.moe_pair(wgu, wd, X[t])
        assert np.array_equal(Y[t], o) and np.array_equal(S[t], s)


def test_ffn_matches_library_matmuls():
    """g, u and y through torch's f64 matmul on the oracle's dequantized
    weights, SiLU from torch: equal within f64 rounding of the sums."""
    H, I, T = 256, 96, 7
    guq, gus, dq, ds = _dense_ffn_weights(64, H, I)
    rng = np.random.default_rng(65)
    X = oracle.x_to_f64(synth.draw_x(rng, T, H, 0.5), "bf16")
    Y, S, A = oracle.ffn(X, guq, gus, dq, ds, I, want_a=True)
    wgu = torch.from_numpy(oracle.dequant_q4(guq, gus, 2 * I, H).astype(np.float64))
    wd = torch.from_numpy(oracle.dequant_q4(dq, ds, H, I).astype(np.float64))
    x = torch.from_numpy(X)
    G = x @ wgu[:I].T
    U = x @ wgu[I:].T
    At = torch.nn.functional.silu(G) * U
    Yt = At @ wd.T
    assert np.allclose(A, At.numpy(), rtol=1e-12, atol=1e-13)
    assert np.all(np.abs(Y - Yt.numpy()) <= 1e-12 * S + 1e-15)


# ---- routing from router logits ---------------------------------------------

def test_route_equal_logits_take_the_lowest_indices_with_equal_weights():
    idx, w = oracle.route(np.zeros((3, 16), np.float32), 5)
    assert idx.tolist() == [[0, 1, 2, 3, 4]] * 3
    assert np.all(w == np.float32(0.2))


def test_route_order_matches_a_stable_library_argsort():
    """The picked experts and their order are the first k of numpy's stable
    argsort of -logits (ties: lower index first), including heavy ties."""
    rng = np.random.default_rng(81)
    lg = rng.integers(-3, 4, (50, 32)).astype(np.float32) * 0.5        # many equal logits
    lg[10] = rng.standard_normal(32).astype(np.float32)
    idx, _ = oracle.route(lg, 8)
    ref = np.argsort(-lg, axis=1, kind="stable")[:, :8]
    assert np.array_equal(idx, ref)


def test_route_weights_closed_form():
    """w_i / w_j = exp(l_i - l_j) for picked experts i, j, and the weights of a
    row sum to 1 (to f32 rounding); two logits ln 3 apart give 3/4 and 1/4."""
    lg = np.array([[0.0, np.log(3.0), -5.0, -6.0]], np.float32)
    idx, w = oracle.route(lg, 2)
    assert idx.tolist() == [[1, 0]]
    e = np.exp(np.float64(lg[0, 1]) - np.float64(lg[0, 0]))
    assert np.allclose(w[0], [e / (1 + e), 1 / (1 + e)], rtol=1e-7)
    rng = np.random.default_rng(82)
    lg = rng.standard_normal((20, 64)).astype(np.float32)
    idx, w = oracle.route(lg, 8)
    assert np.allclose(w.sum(axis=1), 1.0, rtol=4e-7)
    for t in range(20):
        l = lg[t, idx[t]].astype(np.float64)
        assert np.allclose(w[t] / w[t, 0], np.exp(l - l[0]), rtol=1e-6)
        assert np.all(np.diff(l) <= 0)


def test_route_shared_expert_slot():
    """The shared slot is expert E with weight 1 / (1 + exp(-gate)): 1/2 at
    gate 0, 3/4 at gate ln 3; the routed slots ignore the gate column."""
    lg = np.array([[1.0, 2.0, 0.5, 0.0], [1.0, 2.0, 0.5, np.log(3.0)]], np.float32)
    idx, w = oracle.route(lg, 2, shared=True)
    assert idx.tolist() == [[1, 0, 3], [1, 0, 3]]
    assert w[0, 2] == np.float32(0.5) and abs(float(w[1, 2]) - 0.75) < 1e-7
    idx2, w2 = oracle.route(lg[:, :3], 2)
    assert np.array_equal(idx[:, :2], idx2) and np.array_equal(w[:, :2], w2)


def test_route_agrees_with_the_input_recipe():
    """The recipe's own routing of the MoE workload (synth.route_topk, written
    separately from the oracle) picks the same experts with the same weights."""
    m = synth.moe_case(4, T=8, H=256, I=256, E=128, topk=8)
    idx, w = oracle.route(m["logits"], 8)
    assert np.array_equal(idx, m["idx"])
    assert np.allclose(w, m["w"], rtol=1e-6)


# ---- format variants ---------------------------------------------------------

def test_q8b_dequant_is_one_f32_product_per_element():
    """W = RNE_f32(q * s): q * s is exact in f64 (8 + 24 bits), numpy's cast
    to f32 rounds it once; equal to the Q8-row dequantisation when every block
    scale of a row is that row's scale."""
    rng = np.random.default_rng(91)
    q = rng.integers(-128, 128, (7, 96)).astype(np.int8)
    s = rng.uniform(1e-3, 1e-2, (7, 3)).astype(np.float32) * np.where(rng.random((7, 3)) < 0.3, -1, 1).astype(np.float32)
    s[0, 0] = 0.0
    W = oracle.dequant_q8b(q, s)
    ref = (q.astype(np.float64) * np.repeat(s.astype(np.float64), 32, axis=1)).astype(np.float32)
    assert np.array_equal(W.view(np.uint32), ref.view(np.uint32))
    rs = rng.uniform(1e-3, 1e-2, 7).astype(np.float32)
    assert np.array_equal(oracle.dequant_q8b(q, np.repeat(rs[:, None], 3, axis=1)), oracle.dequant_q8row(q, rs))


def test_q4a_dequant_adds_the_group_offset_once():
    """Offsets -0 reproduce the plain Q4 dequantisation bit for bit (adding
    -0 is the IEEE identity, zero signs included; +0 would turn -0 into +0); with
    distinct offsets per group of gk = 2 blocks every element is the f32 sum
    of the exact Q4 value and its group's bf16 offset (numpy f32 addition)."""
    rng = np.random.default_rng(92)
    N, K, gk = 5, 256, 2
    codes, ws = synth.draw_q4(rng, N, K, signed=True)
    wq = oracle.pack_q4(codes)
    zero = np.full((N, K // 32 // gk), 0x8000, np.uint16)
    assert np.array_equal(oracle.dequant_q4a(wq, ws, zero, gk, N, K).view(np.uint32),
                          oracle.dequant_q4(wq, ws, N, K).view(np.uint32))
    off = synth.f32_to_bf16_bits(rng.uniform(-0.1, 0.1, (N, K // 32 // gk)).astype(np.float32))
    W = oracle.dequant_q4a(wq, ws, off, gk, N, K)
    base = (codes.astype(np.float32) - 8) * np.repeat(ws.view(np.float16).astype(np.float32), 32, axis=1)
    m = np.repeat(synth.bf16_bits_to_f32(off), 32 * gk, axis=1)
    assert np.array_equal(W.view(np.uint32), (base + m).astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("T,N,K", [(1, 2, 32), (3, 5, 64)])
def test_q8_2f_vs_exact_rationals(T, N, K):
    rng = np.random.default_rng(93 + K)
    q = rng.integers(-128, 128, (N, K)).astype(np.int8)
    rs = rng.uniform(1e-3, 1e-2, N).astype(np.float16).astype(np.float32)
    col = rng.uniform(0.5, 2.0, K).astype(np.float16).astype(np.float32)
    X = oracle.x_to_f64(synth.draw_x(rng, T, K), "bf16")
    Y, S = oracle.gemm_q8_2f(q, rs, col, X)
    for t in range(T):
        for n in range(N):
            exact = Fraction(float(rs[n])) * sum(Fraction(int(q[n, k])) * Fraction(float(col[k])) * Fraction(X[t, k])
                                                 for k in range(K))
            assert abs(Fraction(Y[t, n]) - exact) <= Fraction(2 ** -50) * Fraction(S[t, n])


def test_q8_2f_with_unit_column_field_is_q8_row():
    rng = np.random.default_rng(94)
    q, rs = synth.draw_q8row(rng, 40, 128)
    X = oracle.x_to_f64(synth.draw_x(rng, 6, 128), "bf16")
    Y, S = oracle.gemm_q8_2f(q, rs, np.ones(128, np.float32), X)
    Yr, Sr = oracle.gemm_q8row(q, rs, X)
    assert np.array_equal(Y, Yr) and np.array_equal(S, Sr)


def test_q8_2f_column_field_scales_activation_columns():
    """Doubling col[k] for one k equals doubling X[:, k] (power of two: exact)."""
    rng = np.random.default_rng(95)
    q, rs = synth.draw_q8row(rng, 16, 64)
    col = rng.uniform(0.5, 2.0, 64).astype(np.float16).astype(np.float32)
    X = oracle.x_to_f64(synth.draw_x(rng, 3, 64), "bf16")
    col2 = col.copy()
    col2[17] *= 2
    X2 = X.copy()
    X2[:, 17] *= 2
    assert np.array_equal(oracle.gemm_q8_2f(q, rs, col2, X)[0], oracle.gemm_q8_2f(q, rs, col, X2)[0])
