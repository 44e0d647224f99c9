"""GPU parity of the format variants against the CPU oracle, through the C
ABI, on both paths (weight streaming for T <= 32, tcgen05 above): Q8 per
32-k block, affine Q4 (a bf16 offset per group of gk blocks) and q8_2f (int8
times a column field, row scale).  Also the Q8/32 decoders bit-exact through
identity activations, as for the other formats."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_weight_02_gb300 as cq
from block_quantized_weight_02_gb300 import pack, synth

from cqtest import DEV, ForcePath, Opt, TORCH_DT, check, to_dev, to_dev_x, traced_kernels, y_host

pytestmark = pytest.mark.gpu

STREAM = [(1, 128, 64), (8, 256, 200), (17, 384, 96), (32, 512, 257)]
TC = [(33, 256, 128), (150, 512, 300), (300, 768, 130)]


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_dev):
    import __graft_entry__
    __graft_entry__.build()


def _q8b_case(seed, T, K, N, xdt):
    rng = np.random.default_rng(seed)
    x = synth.draw_x(rng, T, K, 1.0, xdt)
    q = rng.integers(-127, 128, (N, K)).astype(np.int8)
    s = (rng.uniform(1e-3, 1e-2, (N, K // 32)) * np.where(rng.random((N, K // 32)) < 0.5, -1, 1)).astype(np.float32)
    return x, q, s


@pytest.mark.parametrize("path,T,K,N", [(1, *c) for c in STREAM] + [(2, *c) for c in TC])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
def test_q8b(path, T, K, N, out, xdt):
    x, q, s = _q8b_case(9900 + T + K + N, T, K, N, xdt)
    Y = torch.full((T, N), float("nan"), dtype=TORCH_DT[out], device=DEV)
    ws = torch.empty(cq.cq_gemm_q8b_workspace_bytes(T, K), dtype=torch.uint8, device=DEV)
    with ForcePath(path):
        cq.cq_gemm_q8b(to_dev_x(x, xdt), to_dev(q), to_dev(s), Y, ws)
    assert cq.cq_get_device_error() == 0
    yref, S = oracle.gemm_q8b(q, s, oracle.x_to_f64(x, xdt))
    check(y_host(Y), yref, S, out, f"q8/32 path={path} T={T} K={K} N={N} {xdt}->{out}")


@pytest.mark.parametrize("path,T,kern", [(1, 8, 1), (1, 32, 1), (1, 8, 2), (1, 16, 2), (2, 40, 0), (2, 300, 0)])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
def test_q8b_decoders_bit_exact_identity(path, T, kern, xdt):
    """X[t] = e_{k_t}.  Streaming (kern 1 K-split, 2 row-partitioned): Y =
    RNE_f32(q * s), the oracle's dequantised weight.  tcgen05: Y =
    RNE_fp16(q * RNE_fp16(s)) (numpy's roundings)."""
    K, N = 512, 136
    _, q, s = _q8b_case(9950 + T, 1, K, N, xdt)
    s[0, :] = 0.0
    s[1, :3] = [1.5e-5, -2.0, 0.125]
    kt = 32 * ((5 * np.arange(T) + 3) % (K // 32)) + (13 * np.arange(T) + 3) % 32
    xv = np.zeros((T, K))
    xv[np.arange(T), kt] = 1.0
    x = synth.to_storage(xv, xdt)
    Y = torch.empty(T, N, dtype=torch.float32, device=DEV)
    ws = torch.empty(cq.cq_gemm_q8b_workspace_bytes(T, K), dtype=torch.uint8, device=DEV)
    with ForcePath(path), Opt(cq.CQ_OPT_STREAM_KERNEL, kern):
        cq.cq_gemm_q8b(to_dev_x(x, xdt), to_dev(q), to_dev(s), Y, ws)
    assert cq.cq_get_device_error() == 0
    if path == 1:
        E = oracle.dequant_q8b(q, s)[:, kt].T
    else:
        s16 = s.astype(np.float16).astype(np.float32)
        E = (q.astype(np.float32) * np.repeat(s16, 32, axis=1)).astype(np.float16).astype(np.float32)[:, kt].T
    y = Y.cpu().numpy()
    assert np.array_equal(y == E, np.ones_like(y, bool)), f"{int((y != E).sum())} outputs differ"


@pytest.mark.parametrize("path,T,K,N", [(1, *c) for c in STREAM if c[1] % 256 == 0] + [(1, 5, 768, 130)]
                         + [(2, *c) for c in TC if c[1] % 256 == 0] + [(2, 300, 768, 130)])
@pytest.mark.parametrize("gk", [1, 2, 4])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_q4a(path, T, K, N, gk, out):
    rng = np.random.default_rng(9800 + T + K + N + gk)
    x = synth.draw_x(rng, T, K, 1.0, "bf16")
    codes, ws_ = synth.draw_q4(rng, N, K, signed=True)
    off = synth.f32_to_bf16_bits(rng.uniform(-0.15, 0.15, (N, K // 32 // gk)).astype(np.float32))
    wq = pack.pack_q4(codes)
    Y = torch.full((T, N), float("nan"), dtype=TORCH_DT[out], device=DEV)
    ws = torch.empty(cq.cq_gemm_q4a_workspace_bytes(T, K, N, gk), dtype=torch.uint8, device=DEV)
    with ForcePath(path):
        cq.cq_gemm_q4a(to_dev_x(x, "bf16"), to_dev(wq), to_dev(ws_), to_dev(off), gk, Y, ws)
    assert cq.cq_get_device_error() == 0
    yref, S = oracle.gemm_q4a(wq, ws_, off, gk, N, K, oracle.x_to_f64(x, "bf16"))
    check(y_host(Y), yref, S, out, f"affine q4 path={path} T={T} K={K} N={N} gk={gk} {out}")


@pytest.mark.parametrize("T,bn,ks", [(40, 0, 0), (64, 64, 1), (150, 128, 2), (300, 256, 1), (256, 192, 1)])
@pytest.mark.parametrize("gk", [1, 4])
def test_q4a_tcgen05_decoder_bit_exact_identity(T, bn, ks, gk):
    """X[t] = e_{k_t}.  The tcgen05 decoder takes the bf16 offset to fp16
    (RNE) and forms (nibble - 8) * scale + offset in one fp16 rounding; the
    guard scales the unit row to 2^13 and back exactly, so Y[t][n] =
    RNE_fp16(W4[n][k_t] + RNE_fp16(off)), W4 the oracle's plain Q4 weight
    (exact), the sum taken exactly in f64."""
    K, N = 512, 264
    rng = np.random.default_rng(9600 + T + bn + gk)
    codes = rng.integers(0, 16, (N, K), dtype=np.uint8)
    codes[:, ::7] = 8
    sc = (rng.uniform(0.005, 0.02, (N, K // 32)) * np.where(rng.random((N, K // 32)) < 0.5, -1, 1))
    sc = sc.astype(np.float16).view(np.uint16)
    sc[0, :4] = [0x0000, 0x8000, 0x0001, 0x83FF]   # +-0 and fp16 subnormal scales
    ov = rng.uniform(0.01, 0.15, (N, K // 32 // gk)) * np.where(rng.random((N, K // 32 // gk)) < 0.5, -1, 1)
    ov[1, :3] = [0.0, -0.0, 3.0e-6]                # zeros, and an offset below the fp16 normal range
    off = synth.f32_to_bf16_bits(ov.astype(np.float32))
    wq = pack.pack_q4(codes)
    m16 = synth.bf16_bits_to_f32(off).astype(np.float16).astype(np.float64)
    W = oracle.dequant_q4(wq, sc, N, K).astype(np.float64) + np.repeat(m16, 32 * gk, axis=1)
    E = W.astype(np.float16).astype(np.float32)
    kt = 32 * ((5 * np.arange(T) + 3) % (K // 32)) + (13 * np.arange(T) + 3) % 32
    xv = np.zeros((T, K))
    xv[np.arange(T), kt] = 1.0
    x = synth.to_storage(xv, "bf16")
    Y = torch.empty(T, N, dtype=torch.float32, device=DEV)
    ws = torch.empty(cq.cq_gemm_q4a_workspace_bytes(T, K, N, gk), dtype=torch.uint8, device=DEV)
    with ForcePath(2), Opt(cq.CQ_OPT_TC_BN, bn), Opt(cq.CQ_OPT_TC_KSPLIT, ks):
        cq.cq_gemm_q4a(to_dev_x(x, "bf16"), to_dev(wq), to_dev(sc), to_dev(off), gk, Y, ws)
    assert cq.cq_get_device_error() == 0
    y = Y.cpu().numpy()
    e = E[:, kt].T
    assert np.array_equal(y == e, np.ones_like(y, bool)), f"{int((y != e).sum())} outputs differ"
    nz = e != 0
    assert np.array_equal(y[nz].view(np.uint32), e[nz].view(np.uint32))


@pytest.mark.parametrize("path,T,K,N", [(1, *c) for c in STREAM] + [(2, *c) for c in TC])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
def test_q8_2f(path, T, K, N, out, xdt):
    rng = np.random.default_rng(9700 + T + K + N)
    x = synth.draw_x(rng, T, K, 1.0, xdt)
    q = rng.integers(-127, 128, (N, K)).astype(np.int8)
    rs = rng.uniform(1e-3, 1e-2, N).astype(np.float16).astype(np.float32)
    col = rng.uniform(0.25, 4.0, K).astype(np.float16).astype(np.float32)
    Y = torch.full((T, N), float("nan"), dtype=TORCH_DT[out], device=DEV)
    ws = torch.empty(cq.cq_gemm_q8_2f_workspace_bytes(T, K), dtype=torch.uint8, device=DEV)
    with ForcePath(path):
        cq.cq_gemm_q8_2f(to_dev_x(x, xdt), to_dev(q), to_dev(rs), to_dev(col), Y, ws)
    assert cq.cq_get_device_error() == 0
    yref, S = oracle.gemm_q8_2f(q, rs, col, oracle.x_to_f64(x, xdt))
    check(y_host(Y), yref, S, out, f"q8_2f path={path} T={T} K={K} N={N} {xdt}->{out}")


@pytest.mark.parametrize("T", [1, 8, 16])
@pytest.mark.parametrize("fmt", ["q8b", "q4a", "q8_2f"])
def test_formats_on_the_row_partitioned_kernel(T, fmt, capfd):
    """The format variants at T <= 16 with K a whole number of stages on the
    row-partitioned streaming kernel (Q8/32 decode, the affine addend, q8_2f's
    guarded activations with per-token scales)."""
    with Opt(cq.CQ_OPT_STREAM_KERNEL, 2):
        trace = traced_kernels(capfd, lambda: _formats_rows(T, fmt))
    assert any(l.startswith("cq: rows") for l in trace), trace


def _formats_rows(T, fmt):
    K, N = 1024, 600
    rng = np.random.default_rng(9990 + T)
    x = synth.draw_x(rng, T, K, 1.0, "bf16")
    X = oracle.x_to_f64(x, "bf16")
    Y = torch.full((T, N), float("nan"), dtype=torch.float32, device=DEV)
    if fmt == "q8b":
        _, q, s = _q8b_case(9991 + T, 1, K, N, "bf16")
        ws = torch.empty(cq.cq_gemm_q8b_workspace_bytes(T, K), dtype=torch.uint8, device=DEV)
        cq.cq_gemm_q8b(to_dev_x(x, "bf16"), to_dev(q), to_dev(s), Y, ws)
        yref, S = oracle.gemm_q8b(q, s, X)
    elif fmt == "q4a":
        codes, sc = synth.draw_q4(rng, N, K, signed=True)
        off = synth.f32_to_bf16_bits(rng.uniform(-0.15, 0.15, (N, K // 64)).astype(np.float32))
        wq = pack.pack_q4(codes)
        ws = torch.empty(cq.cq_gemm_q4a_workspace_bytes(T, K, N, 2), dtype=torch.uint8, device=DEV)
        cq.cq_gemm_q4a(to_dev_x(x, "bf16"), to_dev(wq), to_dev(sc), to_dev(off), 2, Y, ws)
        yref, S = oracle.gemm_q4a(wq, sc, off, 2, N, K, X)
    else:
        q = rng.integers(-127, 128, (N, K)).astype(np.int8)
        rs = rng.uniform(1e-3, 1e-2, N).astype(np.float16).astype(np.float32)
        col = rng.uniform(0.25, 4.0, K).astype(np.float16).astype(np.float32)
        ws = torch.empty(cq.cq_gemm_q8_2f_workspace_bytes(T, K), dtype=torch.uint8, device=DEV)
        cq.cq_gemm_q8_2f(to_dev_x(x, "bf16"), to_dev(q), to_dev(rs), to_dev(col), Y, ws)
        yref, S = oracle.gemm_q8_2f(q, rs, col, X)
    assert cq.cq_get_device_error() == 0
    check(y_host(Y), yref, S, "f32", f"{fmt} on the row-partitioned kernel T={T}")
