"""GPU parity of the z-batched Q4 GEMM (one launch over up to four weights
of one shape, each with its own activation and output offset) against the
CPU oracle, job by job, on both paths: the qkv shape (z = 3, one shared X,
outputs side by side), gate/up (z = 2) and four jobs reading two different
activation slices (two guard passes); columns of Y outside the jobs' ranges
stay untouched."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_weight_02_gb300 as cq
from block_quantized_weight_02_gb300 import pack, synth

from cqtest import DEV, TORCH_DT, check, to_dev, y_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_dev):
    import __graft_entry__
    __graft_entry__.build()


def _run(seed, T, K, N, x_offs, y_offs, ldx, ldy, xdt, out):
    rng = np.random.default_rng(seed)
    xv = synth.draw_x(rng, T, ldx, 1.0, xdt)
    ws_list = [synth.draw_q4(rng, N, K, signed=True) for _ in x_offs]
    X = torch.from_numpy(xv.view(np.int16)).view(TORCH_DT[xdt]).to(DEV)
    Y = torch.full((T, ldy), float("nan"), dtype=TORCH_DT[out], device=DEV)
    packed = [(pack.pack_q4(c), s) for c, s in ws_list]
    dev = [(to_dev(q), to_dev(s)) for q, s in packed]
    jobs = [(q, s, xo, yo) for (q, s), xo, yo in zip(dev, x_offs, y_offs)]
    ws = torch.empty(cq.cq_gemm_q4_batched_workspace_bytes(T, K, len(jobs)), dtype=torch.uint8, device=DEV)
    cq.cq_gemm_q4_batched(X, K, jobs, N, Y, ws)
    st = cq.cq_get_device_error()
    assert st == 0, cq.STATUS[st]
    y = y_host(Y)
    Xf = oracle.x_to_f64(xv, xdt)
    covered = np.zeros(ldy, bool)
    for j, ((q, s), xo, yo) in enumerate(zip(packed, x_offs, y_offs)):
        yref, S = oracle.gemm_q4(q, s, N, K, np.ascontiguousarray(Xf[:, xo:xo + K]))
        check(y[:, yo:yo + N], yref, S, out, f"job {j} T={T} K={K} N={N} x_off={xo} y_off={yo}")
        covered[yo:yo + N] = True
    assert np.all(np.isnan(y[:, ~covered])), "columns outside the jobs' outputs were written"


@pytest.mark.parametrize("T", [5, 32, 100, 300])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_batched_qkv_shared_x(T, out):
    K, N = 512, 256
    _run(9300 + T, T, K, N, [0, 0, 0], [0, N, 2 * N], K, 3 * N, "bf16", out)


@pytest.mark.parametrize("T", [8, 200])
def test_batched_gate_up_z2_fp16(T):
    K, N = 768, 384
    _run(9400 + T, T, K, N, [0, 0], [0, N], K, 2 * N, "f16", "f32")


@pytest.mark.parametrize("T", [16, 150])
def test_batched_four_jobs_two_activation_slices_gapped_output(T):
    """Jobs 0, 2 read X[:, 0:K], jobs 1, 3 X[:, K:2K] (two guard passes on the
    tensor-core path); the outputs leave gaps in Y that must stay untouched."""
    K, N = 512, 136
    _run(9500 + T, T, K, N, [0, K, 0, K], [8, 152, 296, 440], 2 * K, 600, "bf16", "f32")


def test_batched_tail_launch(capfd):
    """z = 2 jobs of T = 256, K = 1536, N = 10240 in 256-token tiles: 80 row tiles
    x 2 jobs leave a partial last wave, so the last row tiles of both jobs go to
    a K-split tail launch (trace line "tail"); outputs sampled over every row and
    densely over the last 1024 rows of each job."""
    from cqtest import Opt, sample_positions, traced_kernels
    T, K, N = 256, 1536, 10240
    rng = np.random.default_rng(9600)
    xv = synth.draw_x(rng, T, K, 1.0, "bf16")
    packed = [(pack.pack_q4(c), s) for c, s in (synth.draw_q4(rng, N, K, signed=True) for _ in range(2))]
    X = torch.from_numpy(xv.view(np.int16)).view(TORCH_DT["bf16"]).to(DEV)
    Y = torch.full((T, 2 * N), float("nan"), dtype=torch.float32, device=DEV)
    jobs = [(to_dev(q), to_dev(s), 0, j * N) for j, (q, s) in enumerate(packed)]
    ws = torch.empty(cq.cq_gemm_q4_batched_workspace_bytes(T, K, 2), dtype=torch.uint8, device=DEV)
    with Opt(cq.CQ_OPT_TC_BN, 256):
        trace = traced_kernels(capfd, lambda: cq.cq_gemm_q4_batched(X, K, jobs, N, Y, ws))
    assert any(l.startswith("cq: tcgen05 tail") for l in trace), trace
    assert cq.cq_get_device_error() == 0
    y = y_host(Y)
    Xf = oracle.x_to_f64(xv, "bf16")
    for j, (q, s) in enumerate(packed):
        tn = np.concatenate([sample_positions(T, N, 1500, 9601 + j),
                             np.stack([rng.integers(0, T, 2000), rng.integers(N - 1024, N, 2000)], 1)]).astype(np.int64)
        yref, S = oracle.gemm_q4_sampled(q, s, N, K, Xf, tn)
        check(y[:, j * N:(j + 1) * N][tn[:, 0], tn[:, 1]], yref, S, "f32", f"batched job {j} with a tail launch")
