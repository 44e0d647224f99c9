"""GPU parity of the Q4 / Q8-row GEMMs and the dequantization hooks against
the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_weight_02_gb300 as cq
from block_quantized_weight_02_gb300 import pack, synth

from cqtest import (DEV, ForcePath, check, oracle_q4, oracle_q8, run_q4, run_q8, sample_positions, to_dev,
                    to_dev_x, traced_kernels, y_host)
from test_oracle import _golden_blocks

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_dev):
    import __graft_entry__
    __graft_entry__.build()


# ---- dequantization hooks: bit-exact ------------------------------------

def test_dequant_q4_golden_blocks_bit_exact():
    blocks = _golden_blocks()
    wq = np.stack([np.frombuffer(b[3], np.uint8) for b in blocks])            # one block per row
    ws = np.array([[b[1]] for b in blocks], np.uint16)
    W = torch.empty(len(blocks), 32, dtype=torch.float32, device=DEV)
    cq.cq_dequant_q4(to_dev(wq), to_dev(ws), W)
    ref = oracle.dequant_q4(wq, ws, len(blocks), 32)
    assert np.array_equal(W.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_dequant_q4_random_bit_exact():
    rng = np.random.default_rng(77)
    N, K = 300, 1024
    wq = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
    ws = rng.integers(0, 65536, (N, K // 32), dtype=np.uint32).astype(np.uint16)
    ws[(ws & 0x7C00) == 0x7C00] = 0x3C00        # no inf/NaN scales (IEEE propagation, unpinned)
    ws[:4, :4] = [[0x0000, 0x8000, 0x0001, 0x8001]] * 4
    W = torch.empty(N, K, dtype=torch.float32, device=DEV)
    cq.cq_dequant_q4(to_dev(wq), to_dev(ws), W)
    ref = oracle.dequant_q4(wq, ws, N, K)
    assert np.array_equal(W.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_dequant_q8row_bit_exact():
    rng = np.random.default_rng(78)
    q, rs = synth.draw_q8row(rng, 129, 200)
    q[0, :3] = [-128, 127, 0]
    W = torch.empty(129, 200, dtype=torch.float32, device=DEV)
    cq.cq_dequant_q8row(to_dev(q), to_dev(rs), W)
    assert np.array_equal(W.cpu().numpy().view(np.uint32), oracle.dequant_q8row(q, rs).view(np.uint32))


# ---- small shapes, both paths, full comparison --------------------------

SMALL = [(1, 256, 64), (3, 512, 130), (8, 256, 200), (16, 768, 64), (17, 256, 96), (32, 512, 257)]
LARGE = [(33, 256, 128), (100, 512, 300), (150, 512, 192), (257, 768, 130), (512, 256, 384)]


@pytest.mark.parametrize("T,K,N", SMALL)
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
def test_q4_skinny_small(T, K, N, out, xdt):
    case = synth.gemm_q4_case(1000 + T + K + N, T, K, N, x_dtype=xdt, signed=True)
    with ForcePath(1):
        Y, wq = run_q4(case, out)
    yref, S = oracle_q4(case, wq)
    check(y_host(Y), yref, S, out, f"q4 skinny T={T} K={K} N={N}")


@pytest.mark.parametrize("T,K,N", SMALL + LARGE)
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
def test_q4_tcgen05_small(T, K, N, out, xdt):
    case = synth.gemm_q4_case(2000 + T + K + N, T, K, N, x_dtype=xdt, signed=True)
    with ForcePath(2):
        Y, wq = run_q4(case, out)
    yref, S = oracle_q4(case, wq)
    check(y_host(Y), yref, S, out, f"q4 tcgen05 T={T} K={K} N={N}")


@pytest.mark.parametrize("T,K,N", [(1, 128, 64), (3, 256, 130), (8, 384, 200), (16, 128, 64), (17, 256, 96),
                                   (32, 512, 257)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
def test_q8_skinny_small(T, K, N, out, xdt):
    case = synth.gemm_q8_case(3000 + T + K + N, T, K, N, x_dtype=xdt)
    with ForcePath(1):
        Y = run_q8(case, out)
    yref, S = oracle_q8(case)
    check(y_host(Y), yref, S, out, f"q8 skinny T={T} K={K} N={N}")


@pytest.mark.parametrize("T,K,N", [(1, 128, 64), (17, 256, 96), (33, 128, 128), (100, 384, 300),
                                   (150, 512, 192), (257, 640, 130), (512, 256, 384)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
def test_q8_tcgen05_small(T, K, N, out, xdt):
    case = synth.gemm_q8_case(4000 + T + K + N, T, K, N, x_dtype=xdt)
    with ForcePath(2):
        Y = run_q8(case, out)
    yref, S = oracle_q8(case)
    check(y_host(Y), yref, S, out, f"q8 tcgen05 T={T} K={K} N={N}")


def test_q4_wide_magnitude_rows_guard():
    """Rows spanning 1e-3 .. 2e5 (beyond fp16's range), as in the pages'
    GPU-vs-CPU test ("oxinfer 0.0.5 src/metal.rs", tests module, input())."""
    T, K, N = 32, 512, 192
    rng = np.random.default_rng(5)
    mags = np.array([1e-3, 1.0, 300.0, 2e5])
    xv = (rng.uniform(-0.5, 0.5, (T, K)) * mags[np.arange(T) % 4][:, None])
    case = synth.gemm_q4_case(6, T, K, N)
    case["x"] = synth.to_storage(xv, "bf16")
    for path in (1, 2):
        with ForcePath(path):
            Y, wq = run_q4(case, "f32")
        yref, S = oracle_q4(case, wq)
        check(y_host(Y), yref, S, "f32", f"q4 wide rows path {path}")


def test_q8_wide_magnitude_rows():
    T, K, N = 32, 512, 192
    rng = np.random.default_rng(6)
    mags = np.array([1e-3, 1.0, 300.0, 2e5])
    case = synth.gemm_q8_case(7, T, K, N)
    case["x"] = synth.to_storage(rng.uniform(-0.5, 0.5, (T, K)) * mags[np.arange(T) % 4][:, None], "bf16")
    for path in (1, 2):
        with ForcePath(path):
            Y = run_q8(case, "f32")
        yref, S = oracle_q8(case)
        check(y_host(Y), yref, S, "f32", f"q8 wide rows path {path}")


def test_outputs_overwritten_and_bounds_respected():
    """Y starts as NaN inside a larger buffer; the call fills Y exactly."""
    T, K, N = 29, 512, 200
    case = synth.gemm_q4_case(8, T, K, N)
    for path in (1, 2):
        buf = torch.full((T * N + 4096,), float("nan"), dtype=torch.float32, device=DEV)
        Y = buf[:T * N].view(T, N)
        with ForcePath(path):
            run_q4(case, "f32", Y=Y)
        assert torch.isfinite(Y).all()
        assert torch.isnan(buf[T * N:]).all()


def test_deterministic_repeat():
    case = synth.gemm_q4_case(9, 24, 4096, 512)
    case8 = synth.gemm_q8_case(9, 200, 1024, 512)
    a, _ = run_q4(case, "f32")
    b, _ = run_q4(case, "f32")
    assert torch.equal(a, b)
    c = run_q8(case8, "bf16")
    d = run_q8(case8, "bf16")
    assert torch.equal(c, d)


def test_c1_smallest_q4_case():
    case = synth.c1()
    Y, wq = run_q4(case, "f32")
    yref, S = oracle_q4(case, wq)
    check(y_host(Y), yref, S, "f32", "C1")


# ---- the configured sizes, sampled outputs ------------------------------

def _sampled_q4(case, out, count=3000, seed=0):
    Y, wq = run_q4(case, out)
    tn = sample_positions(case["T"], case["N"], count, seed)
    yref, S = oracle.gemm_q4_sampled(wq, case["scales"], case["N"], case["K"],
                                     oracle.x_to_f64(case["x"], case["x_dtype"]), tn)
    y = y_host(Y)[tn[:, 0], tn[:, 1]]
    return check(y, yref, S, out, f"q4 T={case['T']} K={case['K']} N={case['N']} {out}")


def _sampled_q8(case, out, count=3000, seed=0):
    Y = run_q8(case, out)
    tn = sample_positions(case["T"], case["N"], count, seed)
    yref, S = oracle.gemm_q8_sampled(case["q"], case["rs"], oracle.x_to_f64(case["x"], case["x_dtype"]), tn)
    y = y_host(Y)[tn[:, 0], tn[:, 1]]
    return check(y, yref, S, out, f"q8 T={case['T']} K={case['K']} N={case['N']} {out}")


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_c2_prefill_projection_q4(out):
    _sampled_q4(synth.c2_q4(), out)


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_c2_prefill_projection_q8(out):
    _sampled_q8(synth.c2_q8(), out)


def test_c2_full_output_q4_f32():
    """Every output of the prefill projection (17 GFLOP of f64 on the host)."""
    case = synth.c2_q4()
    Y, wq = run_q4(case, "f32")
    yref, S = oracle_q4(case, wq)
    check(y_host(Y), yref, S, "f32", "C2 q4 full")


def test_c3_denoiser_block():
    gu, dn = synth.c3()
    _sampled_q4(gu, "bf16", count=2000)
    _sampled_q4(dn, "bf16", count=2000)


@pytest.mark.parametrize("T", [1, 8, 32, 128, 512, 2048])
def test_c5_sweep_q4(T):
    for out in ("bf16", "f32"):
        _sampled_q4(synth.c5_q4(T), out, count=1500, seed=T)


@pytest.mark.parametrize("T", [1, 8, 32, 128, 512, 2048])
def test_c5_sweep_q8(T):
    for out in ("bf16", "f32"):
        _sampled_q8(synth.c5_q8(T), out, count=1500, seed=T)


# ---- failure handling without a fault -----------------------------------

def test_wait_timeout_reports_status_and_context_survives():
    case = synth.gemm_q8_case(10, 200, 256, 128)
    old = cq.cq_get_option(cq.CQ_OPT_WAIT_NS)
    try:
        cq.cq_set_option(cq.CQ_OPT_WAIT_NS, 20_000_000)       # 20 ms
        cq.cq_set_option(cq.CQ_OPT_TEST_STALL, 1)             # the next tcgen05 loader issues nothing
        with ForcePath(2):
            X = to_dev_x(case["x"], "bf16")
            Y = torch.empty(200, 128, dtype=torch.float32, device=DEV)
            cq.cq_gemm_q8row(X, to_dev(case["q"]), to_dev(case["rs"]), Y)
        assert cq.cq_get_device_error() == 8                   # CQ_ERR_TIMEOUT
    finally:
        cq.cq_set_option(cq.CQ_OPT_WAIT_NS, old)
        cq.cq_set_option(cq.CQ_OPT_TEST_STALL, 0)
    Y = run_q8(case, "f32")                                   # the context is still usable
    yref, S = oracle_q8(case)
    check(y_host(Y), yref, S, "f32", "after timeout")


class _Opt:
    """Context manager setting one library option for the duration."""

    def __init__(self, opt, value):
        self.opt, self.value = opt, value

    def __enter__(self):
        self.old = cq.cq_get_option(self.opt)
        cq.cq_set_option(self.opt, self.value)

    def __exit__(self, *a):
        cq.cq_set_option(self.opt, self.old)


@pytest.mark.parametrize("am", [1, 2])
@pytest.mark.parametrize("ks", [1, 2])
@pytest.mark.parametrize("bn", [32, 64, 128, 256])
def test_tcgen05_ksplit_token_tiles_and_operand_modes(ks, bn, am):
    """Every token tile, K split (one CTA, or two CTAs of a cluster whose
    partial sums are exchanged in shared memory) and placement of the decoded
    weight operand (1 shared memory, 2 tensor memory), on shapes with a
    ragged weight-row tile (N=300) and a ragged token tile."""
    case4 = synth.gemm_q4_case(5000 + ks + bn, 150, 512, 300, x_dtype="bf16", signed=True)
    case8 = synth.gemm_q8_case(6000 + ks + bn, 150, 512, 300, x_dtype="bf16")
    with ForcePath(2), _Opt(cq.CQ_OPT_TC_KSPLIT, ks), _Opt(cq.CQ_OPT_TC_BN, bn), _Opt(cq.CQ_OPT_TC_AMODE, am):
        Y4, wq = run_q4(case4, "f32")
        Y8 = run_q8(case8, "bf16")
    yref, S = oracle_q4(case4, wq)
    check(y_host(Y4), yref, S, "f32", f"q4 ks={ks} bn={bn} am={am}")
    yref8, S8 = oracle_q8(case8)
    check(y_host(Y8), yref8, S8, "bf16", f"q8 ks={ks} bn={bn} am={am}")


@pytest.mark.parametrize("K", [128, 384, 640])
@pytest.mark.parametrize("bn", [32, 64, 128, 256])
def test_tcgen05_q8_short_last_round(K, bn):
    """Q8-row K (a multiple of 128) whose 64-k stages do not fill the last
    round of decoded slots handed to the MMA thread: the decoder groups without
    a stage in it still complete the round."""
    case8 = synth.gemm_q8_case(7300 + K + bn, 200, K, 256, x_dtype="bf16")
    with ForcePath(2), _Opt(cq.CQ_OPT_TC_BN, bn), _Opt(cq.CQ_OPT_TC_KSPLIT, 1):
        Y8 = run_q8(case8, "f32")
    yref8, S8 = oracle_q8(case8)
    check(y_host(Y8), yref8, S8, "f32", f"q8 K={K} bn={bn}")


@pytest.mark.parametrize("bn", [32, 128, 192, 256])
@pytest.mark.parametrize("ks", [1, 2])
@pytest.mark.parametrize("pair", [1, 2])
def test_tcgen05_cta_pairs(ks, pair, bn):
    """32-, 128-, 192- and 256-column tiles with neighbouring weight-row tiles
    sharing one 256-row MMA on a CTA pair (192 columns: pairs only, no K split) (each CTA decoding its rows into its own tensor memory and
    loading half of the activation rows) against the unpaired kernel and the
    oracle: an even number of row tiles with a ragged last one (N=468), a
    ragged token tile, both weight formats and both activation types."""
    case4 = synth.gemm_q4_case(7100 + ks, 300, 512, 468, x_dtype="bf16", signed=True)
    case8 = synth.gemm_q8_case(7200 + ks, 300, 512, 468, x_dtype="f16")
    case8b = synth.gemm_q8_case(7250 + ks, 300, 512, 468, x_dtype="bf16")
    with ForcePath(2), _Opt(cq.CQ_OPT_TC_KSPLIT, ks), _Opt(cq.CQ_OPT_TC_BN, bn), _Opt(cq.CQ_OPT_TC_PAIR, pair):
        Y4, wq = run_q4(case4, "f32")
        Y8 = run_q8(case8, "bf16")
        Y8b = run_q8(case8b, "f32")
    yref, S = oracle_q4(case4, wq)
    check(y_host(Y4), yref, S, "f32", f"q4 ks={ks} pair={pair} bn={bn}")
    yref8, S8 = oracle_q8(case8)
    check(y_host(Y8), yref8, S8, "bf16", f"q8 f16 ks={ks} pair={pair} bn={bn}")
    yref8b, S8b = oracle_q8(case8b)
    check(y_host(Y8b), yref8b, S8b, "f32", f"q8 bf16 ks={ks} pair={pair} bn={bn}")


@pytest.mark.parametrize("T", [1, 8, 17, 32])
def test_q4_weight_streaming_fp16_activations_at_the_range_edges(T):
    """The weight-streaming path multiplies the caller's fp16 activations as
    given (no guard): values near the fp16 maximum, subnormals and zeros,
    with exact nibble - 8 weights, every product exact in f32."""
    K, N = 512, 192
    rng = np.random.default_rng(40 + T)
    xv = rng.uniform(-1.0, 1.0, (T, K))
    xv[:, 0::7] *= 60000.0           # near the fp16 maximum (65504)
    xv[:, 3::11] *= 2.0 ** -20       # fp16 subnormals
    xv[:, 5::13] = 0.0
    case = synth.gemm_q4_case(9, T, K, N, x_dtype="f16", signed=True)
    case["x"] = synth.to_storage(xv, "f16")
    with ForcePath(1):
        Y, wq = run_q4(case, "f32")
    yref, S = oracle_q4(case, wq)
    check(y_host(Y), yref, S, "f32", f"q4 streaming fp16 edges T={T}")


# ---- weight-streaming Q4: partition shapes, workspace contents, graph replay ----

@pytest.mark.parametrize("T,K,N", [(1, 8192, 130), (8, 4096, 64), (8, 256, 1000), (16, 2048, 600),
                                   (32, 1024, 777), (5, 768, 129), (1, 256, 40000)])
def test_q4_streaming_partition_shapes(T, K, N):
    """Shapes that split a row block's K over a cluster (few rows, long K), leave a
    ragged last row block, give a CTA a single stage (K = 256), or make row blocks
    outnumber two CTAs per SM (no K split); the result is compared element by
    element with the oracle."""
    case = synth.gemm_q4_case(2000 + T + K + N, T, K, N, x_dtype="bf16", signed=True)
    with ForcePath(1):
        Y, wq = run_q4(case, "f32")
    yref, S = oracle_q4(case, wq)
    check(y_host(Y), yref, S, "f32", f"q4 streaming T={T} K={K} N={N}")


def test_q4_streaming_workspace_contents_and_graph_replay():
    """The workspace may hold anything: filled with 0xFF bytes, with random bytes,
    or with the guard copy a T > 32 call leaves in it, the weight-streaming result
    is the same bit for bit; so is every replay of a captured CUDA graph."""
    T, K, N = 8, 2048, 520
    case = synth.gemm_q4_case(77, T, K, N, x_dtype="bf16", signed=True)
    wq = pack.pack_q4(case["codes"])
    X = to_dev_x(case["x"], "bf16")
    Wq, Ws = to_dev(wq), to_dev(case["scales"])
    big = synth.gemm_q4_case(78, 64, K, N, x_dtype="bf16", signed=True)
    Xb = to_dev_x(big["x"], "bf16")
    Yb = torch.empty(64, N, dtype=torch.float32, device=DEV)
    nbytes = max(cq.cq_gemm_q4_workspace_bytes(T, K), cq.cq_gemm_q4_workspace_bytes(64, K))
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=DEV)
    Y = torch.empty(T, N, dtype=torch.float32, device=DEV)
    with ForcePath(0):
        cq.cq_gemm_q4(X, Wq, Ws, Y, ws)
        ref = Y.clone()
        yref, S = oracle_q4(case, wq)
        check(y_host(ref), yref, S, "f32", "q4 streaming, workspace of 0xFF bytes")
        ws.copy_(torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=DEV))
        Y.zero_()
        cq.cq_gemm_q4(X, Wq, Ws, Y, ws)
        assert torch.equal(Y, ref)
        cq.cq_gemm_q4(Xb, Wq, Ws, Yb, ws)          # the guard pass writes over the workspace
        Y.zero_()
        cq.cq_gemm_q4(X, Wq, Ws, Y, ws)
        assert torch.equal(Y, ref)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            cq.cq_gemm_q4(X, Wq, Ws, Y, ws)          # warm up on the capture stream
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cq.cq_gemm_q4(X, Wq, Ws, Y, ws)
        for _ in range(3):
            Y.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert cq.cq_get_device_error() == 0
            assert torch.equal(Y, ref)


# ---- the GEMMs' own decoders, bit-exact through identity activations ----
# Row t of X is the unit vector at column k_t, so output (t, n) is the single
# product W[n][k_t] * 1 plus exact zeros.  On the weight-streaming path every
# product is exact and the block scale multiplies the f32 result of its
# block, so Y[t][n] is the oracle's dequantized weight itself (one exact f32
# product).  On the tcgen05 path the decoder rounds (q - 8) * scale once to
# fp16, the guard scales the unit row to 2^13 and back, so Y[t][n] is the
# fp16 rounding (RNE) of the oracle's weight.  The only freedom is the sign
# of a zero result, which a sum does not carry, so values are compared with
# == (+0 == -0) and every nonzero value is then equal bit for bit.

_SPECIAL_SCALES = np.array([0x0000, 0x8000, 0x0001, 0x8001, 0x03FF, 0x83FF, 0x0400, 0x3C00, 0xBC00, 0x2E66],
                           np.uint16)


def _decoder_case(seed, N, K, big_scales):
    """Codes over 0..15 with nibble 8 (zero) on every 7th column, signed fp16
    block scales with +-0, subnormal, smallest normal and unit scales mixed in
    (and, where no fp16 rounding of the weight follows, the largest finite)."""
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, (N, K), dtype=np.uint8)
    codes[:, ::7] = 8
    mag = rng.uniform(0.005, 0.02, (N, K // 32)) * np.where(rng.integers(0, 2, (N, K // 32)) == 1, -1.0, 1.0)
    scales = mag.astype(np.float16).view(np.uint16)
    specials = np.concatenate([_SPECIAL_SCALES, np.array([0x7BFF, 0xFBFF], np.uint16)]) if big_scales \
        else _SPECIAL_SCALES
    m = rng.random(scales.shape) < 0.25
    scales[m] = rng.choice(specials, int(m.sum()))
    return codes, scales


def _unit_rows(T, K, xdt, shift):
    """X[t] = e_{k_t}: block (5 t + shift) mod K/32, position (13 t + shift) mod 32
    (every position of a 32-k block once per 32 rows)."""
    nb = K // 32
    kt = 32 * ((5 * np.arange(T) + shift) % nb) + (13 * np.arange(T) + shift) % 32
    x = np.zeros((T, K))
    x[np.arange(T), kt] = 1.0
    return synth.to_storage(x, xdt), kt


def _assert_values_equal(Y, E, what):
    y = Y.cpu().numpy()
    eq = y == E
    assert eq.all(), (f"{what}: {int((~eq).sum())} of {eq.size} outputs differ, first at "
                      f"{np.argwhere(~eq)[0]}: {y[tuple(np.argwhere(~eq)[0])]!r} vs {E[tuple(np.argwhere(~eq)[0])]!r}")
    nz = E != 0
    assert np.array_equal(y[nz].view(np.uint32), E[nz].astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("T", [1, 8, 16, 32])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
@pytest.mark.parametrize("kern", [1, 2])
def test_q4_streaming_decoder_bit_exact_identity(T, xdt, kern):
    """Both weight-streaming kernels (1 K-split, 2 row-partitioned)."""
    N, K = 300, 1024
    codes, scales = _decoder_case(8100 + T, N, K, big_scales=True)
    wq = pack.pack_q4(codes)
    W = oracle.dequant_q4(wq, scales, N, K)
    for shift in (0, 7):
        x, kt = _unit_rows(T, K, xdt, shift)
        Y = torch.empty(T, N, dtype=torch.float32, device=DEV)
        with ForcePath(1), _Opt(cq.CQ_OPT_STREAM_KERNEL, kern):
            cq.cq_gemm_q4(to_dev_x(x, xdt), to_dev(wq), to_dev(scales), Y,
                          torch.empty(cq.cq_gemm_q4_workspace_bytes(T, K), dtype=torch.uint8, device=DEV))
        assert cq.cq_get_device_error() == 0
        _assert_values_equal(Y, W[:, kt].T, f"q4 streaming decode kernel={kern} T={T} {xdt} shift={shift}")


@pytest.mark.parametrize("T,bn,ks", [(40, 0, 0), (64, 64, 1), (150, 128, 2), (300, 256, 1), (300, 256, 2),
                                     (256, 192, 1)])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
def test_q4_tcgen05_decoder_bit_exact_identity(T, bn, ks, xdt):
    N, K = 512, 512
    codes, scales = _decoder_case(8200 + T + bn, N, K, big_scales=False)
    wq = pack.pack_q4(codes)
    W16 = oracle.dequant_q4(wq, scales, N, K).astype(np.float16).astype(np.float32)   # numpy RNE to fp16
    x, kt = _unit_rows(T, K, xdt, 3)
    Y = torch.empty(T, N, dtype=torch.float32, device=DEV)
    with ForcePath(2), _Opt(cq.CQ_OPT_TC_BN, bn), _Opt(cq.CQ_OPT_TC_KSPLIT, ks):
        cq.cq_gemm_q4(to_dev_x(x, xdt), to_dev(wq), to_dev(scales), Y,
                      torch.empty(cq.cq_gemm_q4_workspace_bytes(T, K), dtype=torch.uint8, device=DEV))
    assert cq.cq_get_device_error() == 0
    _assert_values_equal(Y, W16[:, kt].T, f"q4 tcgen05 decode T={T} bn={bn} ks={ks} {xdt}")


@pytest.mark.parametrize("path,T,bn,ks", [(1, 8, 0, 0), (1, 32, 0, 0), (3, 8, 0, 0), (3, 32, 0, 0),
                                          (2, 64, 64, 1), (2, 300, 256, 2), (2, 200, 128, 1)])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
def test_q8_decoders_bit_exact_identity(path, T, bn, ks, xdt):
    """Q8-row: int8 -> the activation type exactly, the row scale on the f32
    sum: Y[t][n] = RNE_f32(q[n][k_t] * rs[n]), the oracle's dequantized weight."""
    N, K = 260, 512
    rng = np.random.default_rng(8300 + T)
    q, rs = synth.draw_q8row(rng, N, K)
    q[0, :] = -128
    q[1, :] = 127
    q[2, ::3] = 0
    W = oracle.dequant_q8row(q, rs)
    x, kt = _unit_rows(T, K, xdt, 11)
    Y = torch.empty(T, N, dtype=torch.float32, device=DEV)
    # path 1: the K-split streaming kernel, 3: the row-partitioned one, 2: tcgen05
    with ForcePath(min(path, 2) if path != 3 else 1), _Opt(cq.CQ_OPT_STREAM_KERNEL, 2 if path == 3 else 1), \
            _Opt(cq.CQ_OPT_TC_BN, bn), _Opt(cq.CQ_OPT_TC_KSPLIT, ks):
        cq.cq_gemm_q8row(to_dev_x(x, xdt), to_dev(q), to_dev(rs), Y)
    assert cq.cq_get_device_error() == 0
    _assert_values_equal(Y, W[:, kt].T, f"q8 decode path={path} T={T} bn={bn} ks={ks} {xdt}")


# ---- C3 with f32 outputs: the strict bound on the largest shapes ---------

def test_c3_denoiser_block_f32():
    gu, dn = synth.c3()
    _sampled_q4(gu, "f32", count=2000, seed=3)
    _sampled_q4(dn, "f32", count=2000, seed=4)


# ---- the row-partitioned weight-streaming kernel (T <= 16) -------------------

@pytest.mark.parametrize("T", [1, 3, 8, 9, 16, 17, 32])
@pytest.mark.parametrize("K,N", [(512, 8), (1024, 100), (2048, 1001), (4096, 2500), (512, 20000)])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
def test_q4_rows_kernel(T, K, N, xdt, capfd):
    """Units of 8 weight rows spread over one CTA per SM (ragged last unit, a
    tile with one unit, fewer units than SMs, several passes of eight units per
    CTA at N = 20000), the whole K per CTA; f32 output for even T, bf16 for odd."""
    out = "f32" if T % 2 == 0 else "bf16"
    case = synth.gemm_q4_case(8400 + T + K + N, T, K, N, x_dtype=xdt, signed=True)
    res = {}
    with ForcePath(1), _Opt(cq.CQ_OPT_STREAM_KERNEL, 2):
        trace = traced_kernels(capfd, lambda: res.update(r=run_q4(case, out)))
    assert any(l.startswith("cq: rows") for l in trace), trace
    Y, wq = res["r"]
    yref, S = oracle_q4(case, wq)
    check(y_host(Y), yref, S, out, f"q4 rows T={T} K={K} N={N} {xdt}")


@pytest.mark.parametrize("T", [1, 8, 16, 25, 32])
@pytest.mark.parametrize("K,N", [(512, 8), (1536, 300), (2048, 1001), (512, 20000)])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
def test_q8_rows_kernel(T, K, N, xdt, capfd):
    case = synth.gemm_q8_case(8500 + T + K + N, T, K, N, x_dtype=xdt)
    res = {}
    with ForcePath(1), _Opt(cq.CQ_OPT_STREAM_KERNEL, 2):
        trace = traced_kernels(capfd, lambda: res.update(Y=run_q8(case, "f32")))
    assert any(l.startswith("cq: rows") for l in trace), trace
    yref, S = oracle_q8(case)
    check(y_host(res["Y"]), yref, S, "f32", f"q8 rows T={T} K={K} N={N} {xdt}")


def test_small_t_kernels_agree():
    """The row-partitioned and the K-split cluster kernels on the same inputs:
    both within the bound of the oracle (the sums run in different orders)."""
    case = synth.gemm_q4_case(8600, 8, 4096, 1000, x_dtype="bf16", signed=True)
    outs = []
    for kern in (1, 2):
        with ForcePath(1), _Opt(cq.CQ_OPT_STREAM_KERNEL, kern):
            Y, wq = run_q4(case, "f32")
        outs.append(y_host(Y))
    yref, S = oracle_q4(case, wq)
    for y in outs:
        check(y, yref, S, "f32", "small-T kernels")
    assert np.all(np.abs(outs[0] - outs[1]) <= 4e-3 * S + 2e-6)


# ---- a partial last wave moved into a K-split launch --------------------------

@pytest.mark.parametrize("fmt", ["q4", "q8"])
def test_tcgen05_tail_launch(fmt, capfd):
    """T = 256, K = 1536, N = 20480 with 256-column tiles: 160 row tiles on the
    GPU's SMs leave a partial last wave, whose row tiles go to a second launch
    with K split over a cluster (trace line "tail").  Outputs sampled over all
    rows and, more densely, over the last 2048 rows (the tail's and its
    neighbours')."""
    T, K, N = 256, 1536, 20480
    case = (synth.gemm_q4_case(8700, T, K, N) if fmt == "q4" else synth.gemm_q8_case(8701, T, K, N))
    res = {}
    with ForcePath(2), _Opt(cq.CQ_OPT_TC_BN, 256):
        run = (lambda: res.update(r=run_q4(case, "f32"))) if fmt == "q4" else (lambda: res.update(r=(run_q8(case, "f32"), None)))
        trace = traced_kernels(capfd, run)
    assert any(l.startswith("cq: tcgen05 tail") for l in trace), trace
    Y, wq = res["r"]
    rng = np.random.default_rng(8702)
    tn = np.concatenate([sample_positions(T, N, 2000, 8703),
                         np.stack([rng.integers(0, T, 3000), rng.integers(N - 2048, N, 3000)], 1)]).astype(np.int64)
    X = oracle.x_to_f64(case["x"], case["x_dtype"])
    if fmt == "q4":
        yref, S = oracle.gemm_q4_sampled(wq, case["scales"], N, K, X, tn)
    else:
        yref, S = oracle.gemm_q8_sampled(case["q"], case["rs"], X, tn)
    check(y_host(Y)[tn[:, 0], tn[:, 1]], yref, S, "f32", f"{fmt} tcgen05 with a K-split tail launch")
