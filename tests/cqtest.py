"""Shared helpers of the GPU parity tests: upload seeded inputs, run the
C-ABI entry points, compare with the CPU oracle under the acceptance bound
|y - y_ref| <= 2e-3 * sum_k |w_k x_k| + 1e-6 per element and relative
Frobenius error <= 1e-3, applied to the value before a bf16 output's
mandatory final rounding (see check())."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import block_quantized_weight_02_gb300 as cq
from block_quantized_weight_02_gb300 import pack

DEV = "cuda:0"
TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def to_dev_x(x_bits: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).view(TORCH_DT[dtype]).to(DEV)


def to_dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(DEV)


def y_host(Y: torch.Tensor) -> np.ndarray:
    return Y.float().cpu().numpy().astype(np.float64)


def half_ulp_bf16(y: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |y| (y already a bf16 value)."""
    a = np.abs(y)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(np.maximum(e, -126) - 8), 2.0**-134)


def check(y: np.ndarray, yref: np.ndarray, S: np.ndarray, out_dtype: str, what: str = ""):
    """Acceptance: the computed value before the output's own rounding is
    within |err| <= 2e-3*S + 1e-6 per element and relative Frobenius <= 1e-3
    of the f64 reference.

    An f32 output's rounding (2^-24 relative) is far inside that, so y itself
    is tested.  A bf16 output y stands for every value in its rounding box
    [y - r, y + r] (r = half a bf16 ulp at y), and the bound holds for the
    unrounded value exactly when some value in that box meets it: the test
    takes d = max(|y - yref| - r, 0), the distance from yref to the box, and
    requires d <= 2e-3*S + 1e-6 per element and ||d|| <= 1e-3 ||yref||.

    For bf16 it also compares y with RNE_bf16(yref), the oracle's own
    rounding: a value v within b of yref rounds to a bf16 number at most
    b + r + r' from it (r' the half ulp at RNE_bf16(yref)), so wherever the
    element bound b is below half an ulp the two are equal or adjacent bf16
    numbers.  "One ulp everywhere" is not implied by the bound: where |y| is
    small against S (cancellation) b spans many ulps of y."""
    bound = 2e-3 * S + 1e-6
    nref = max(np.linalg.norm(yref), 1e-300)
    if out_dtype == "bf16":
        r = half_ulp_bf16(y)
        d = np.maximum(np.abs(y - yref) - r, 0.0)
        z = oracle.x_to_f64(oracle.f64_to_bf16(yref), "bf16")
        co = np.abs(y - z) <= bound + r + half_ulp_bf16(z)
    else:
        d = np.abs(y - yref)
        co = np.ones(y.shape, bool)
    bad = d > bound
    fro = np.linalg.norm(d) / nref
    if bad.any() or not np.all(np.isfinite(y)) or fro > 1e-3 or not co.all():
        i = int(np.argmax(d / bound))
        raise AssertionError(f"{what}: {int(bad.sum())} elements over the bound (worst ratio "
                             f"{float((d / bound).flat[i]):.3g} at {np.unravel_index(i, d.shape)}: "
                             f"y={y.flat[i]!r} ref={yref.flat[i]!r} S={S.flat[i]!r}), rel Frobenius {fro:.3g} "
                             f"(bound 1e-3), {int((~co).sum())} bf16 outputs away from the oracle's rounding")
    return float(np.max(d / bound)), float(fro)


def run_q4(case, out_dtype="f32", Y=None):
    T, K, N = case["T"], case["K"], case["N"]
    wq = pack.pack_q4(case["codes"])
    X = to_dev_x(case["x"], case["x_dtype"])
    Wq = to_dev(wq)
    Ws = to_dev(case["scales"])
    if Y is None:
        Y = torch.empty(T, N, dtype=TORCH_DT[out_dtype], device=DEV)
    ws = torch.empty(max(cq.cq_gemm_q4_workspace_bytes(T, K), 1), dtype=torch.uint8, device=DEV)
    cq.cq_gemm_q4(X, Wq, Ws, Y, ws)
    st = cq.cq_get_device_error()
    assert st == 0, cq.STATUS[st]
    return Y, wq


def run_q8(case, out_dtype="f32", Y=None):
    T, K, N = case["T"], case["K"], case["N"]
    X = to_dev_x(case["x"], case["x_dtype"])
    if Y is None:
        Y = torch.empty(T, N, dtype=TORCH_DT[out_dtype], device=DEV)
    cq.cq_gemm_q8row(X, to_dev(case["q"]), to_dev(case["rs"]), Y)
    st = cq.cq_get_device_error()
    assert st == 0, cq.STATUS[st]
    return Y


def oracle_q4(case, wq):
    X = oracle.x_to_f64(case["x"], case["x_dtype"])
    return oracle.gemm_q4(wq, case["scales"], case["N"], case["K"], X)


def oracle_q8(case):
    X = oracle.x_to_f64(case["x"], case["x_dtype"])
    return oracle.gemm_q8row(case["q"], case["rs"], X)


def sample_positions(T, N, count, seed):
    """Corners, edges and random (t, n) positions."""
    rng = np.random.default_rng(seed)
    fixed = [(0, 0), (0, N - 1), (T - 1, 0), (T - 1, N - 1), (T // 2, N // 2)]
    rnd = np.stack([rng.integers(0, T, count), rng.integers(0, N, count)], axis=1)
    return np.concatenate([np.array(fixed, np.int64), rnd.astype(np.int64)])


class ForcePath:
    """Context manager: route GEMMs through one path (1 weight-streaming, 2 tcgen05)."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        self.old = cq.cq_get_option(cq.CQ_OPT_FORCE_PATH)
        cq.cq_set_option(cq.CQ_OPT_FORCE_PATH, self.path)

    def __exit__(self, *a):
        cq.cq_set_option(cq.CQ_OPT_FORCE_PATH, self.old)


class Opt:
    """Context manager setting one library option for the duration."""

    def __init__(self, opt, value):
        self.opt, self.value = opt, value

    def __enter__(self):
        self.old = cq.cq_get_option(self.opt)
        cq.cq_set_option(self.opt, self.value)

    def __exit__(self, *a):
        cq.cq_set_option(self.opt, self.old)


def traced_kernels(capfd, fn):
    """Runs fn() with the library's launch trace on; returns the trace lines
    (the library writes them to the process's standard error)."""
    capfd.readouterr()
    with Opt(cq.CQ_OPT_TRACE, 1):
        fn()
        torch.cuda.synchronize()
    return [l for l in capfd.readouterr().err.splitlines() if l.startswith("cq:")]
