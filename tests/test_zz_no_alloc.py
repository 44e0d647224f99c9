"""cq_gemm_q4_noalloc: the Q4 GEMM for callers that cannot allocate device
memory (a plugin inside a framework that owns all device allocations, a
fixed memory budget, a loop that must not call cudaMalloc).  It keeps its
scratch in a fixed array inside the library instead of a caller workspace.

These tests call it through the C ABI on two calls in a row with different
inputs, the larger call first, so stale contents of the shared array from the
first call would show in the second.  Each output must equal cq_gemm_q4's
(the workspace version, the same deterministic kernels) bit for bit and meet
the acceptance bound against the CPU oracle.  The file is collected last."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_weight_02_gb300 as cq
from block_quantized_weight_02_gb300 import pack, synth

from cqtest import DEV, TORCH_DT, check, to_dev, to_dev_x, y_host


@pytest.fixture(scope="module")
def built():
    import __graft_entry__
    __graft_entry__.build()


def _inputs(case):
    wq = pack.pack_q4(case["codes"])
    return to_dev_x(case["x"], case["x_dtype"]), to_dev(wq), to_dev(case["scales"]), wq


def _with_workspace(case, out):
    X, Wq, Ws, _ = _inputs(case)
    Y = torch.empty(case["T"], case["N"], dtype=TORCH_DT[out], device=DEV)
    ws = torch.empty(cq.cq_gemm_q4_workspace_bytes(case["T"], case["K"]), dtype=torch.uint8, device=DEV)
    cq.cq_gemm_q4(X, Wq, Ws, Y, ws)
    assert cq.cq_get_device_error() == 0
    return Y


def _without_workspace(case, out):
    X, Wq, Ws, _ = _inputs(case)
    Y = torch.full((case["T"], case["N"]), float("nan"), dtype=TORCH_DT[out], device=DEV)
    assert cq.lib().cq_set_option(99, 0) != 0              # leaves a message behind
    cq.cq_gemm_q4_noalloc(X, Wq, Ws, Y)
    assert cq.cq_last_error() == ""
    assert cq.cq_get_device_error() == 0
    return Y


@pytest.mark.gpu
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
@pytest.mark.parametrize("shapes", [
    [(24, 1024, 300, "f32"), (9, 512, 200, "bf16")],       # weight-streaming path, two calls
    [(333, 768, 130, "bf16"), (200, 512, 300, "f32")],     # tcgen05 path: the larger call first
])
def test_noalloc_matches_workspace_entry_point_two_calls(cuda_dev, built, shapes, xdt):
    for i, (T, K, N, out) in enumerate(shapes):
        case = synth.gemm_q4_case(900 + 10 * i + T, T, K, N, x_dtype=xdt, signed=True)
        y_ws = _with_workspace(case, out)
        y = _without_workspace(case, out)
        assert torch.equal(y, y_ws), f"noalloc call {i + 1} differs from cq_gemm_q4"
        X = oracle.x_to_f64(case["x"], xdt)
        yref, S = oracle.gemm_q4(pack.pack_q4(case["codes"]), case["scales"], N, K, X)
        check(y_host(y), yref, S, out, f"noalloc call {i + 1} T={T} K={K} N={N} {xdt}")


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_dev, built):
    T, K = 2048, 8192                 # 32 MiB of fp16 activations > the fixed scratch
    assert T * K * 2 > 16 * 1024 * 1024
    X = torch.zeros(T, K, dtype=torch.bfloat16, device=DEV)
    Wq = torch.zeros(64, K // 2, dtype=torch.uint8, device=DEV)
    Ws = torch.zeros(64, K // 32, dtype=torch.int16, device=DEV)
    Y = torch.full((T, 64), 5.0, dtype=torch.float32, device=DEV)
    st = cq.cq_gemm_q4_noalloc(X, Wq, Ws, Y, raise_on_error=False)
    assert st == 3                    # CQ_ERR_SHAPE, nothing launched
    assert "exceeds" in cq.cq_last_error()
    torch.cuda.synchronize()
    assert torch.all(Y == 5.0)
