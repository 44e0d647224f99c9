"""GPU parity of the dense FFN chain (gate/up GEMM with SwiGLU in its
epilogue, then the down GEMM) against the CPU oracle's f64 chain, through the
C ABI: small shapes and every tile option of the gate/up kernel in full, and
the denoiser block's own weights at its full size (T=1024, H=3072,
I=12288), every output compared."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_weight_02_gb300 as cq
from block_quantized_weight_02_gb300 import pack, synth

from cqtest import DEV, TORCH_DT, check, to_dev, to_dev_x, y_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_dev):
    import __graft_entry__
    __graft_entry__.build()


class _Opt:
    def __init__(self, opt, value):
        self.opt, self.value = opt, value

    def __enter__(self):
        self.old = cq.cq_get_option(self.opt)
        cq.cq_set_option(self.opt, self.value)

    def __exit__(self, *a):
        cq.cq_set_option(self.opt, self.old)


def _case(seed, T, H, I, xdt="bf16", x_std=1.0):
    rng = np.random.default_rng(seed)
    x = synth.draw_x(rng, T, H, x_std, xdt)
    gc, gs = synth.draw_q4(rng, 2 * I, H, signed=True)
    dc, ds = synth.draw_q4(rng, H, I, signed=True)
    return {"x": x, "x_dtype": xdt, "guq": pack.pack_q4(gc), "gus": gs, "dq": pack.pack_q4(dc), "ds": ds,
            "T": T, "H": H, "I": I}


def _run(c, out):
    T, H, I = c["T"], c["H"], c["I"]
    Y = torch.full((T, H), float("nan"), dtype=TORCH_DT[out], device=DEV)
    ws = torch.empty(cq.cq_ffn_q4_workspace_bytes(T, H, I), dtype=torch.uint8, device=DEV)
    cq.cq_ffn_q4(to_dev_x(c["x"], c["x_dtype"]), to_dev(c["guq"]), to_dev(c["gus"]), to_dev(c["dq"]),
                 to_dev(c["ds"]), Y, ws)
    st = cq.cq_get_device_error()
    assert st == 0, cq.STATUS[st]
    return Y


def _oracle(c):
    return oracle.ffn(oracle.x_to_f64(c["x"], c["x_dtype"]), c["guq"], c["gus"], c["dq"], c["ds"], c["I"])


@pytest.mark.parametrize("T,H,I", [(1, 256, 256), (7, 512, 256), (33, 256, 512), (150, 768, 256), (300, 256, 768)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
def test_ffn_small(T, H, I, out, xdt):
    c = _case(9000 + T + H + I, T, H, I, xdt)
    Y = _run(c, out)
    yref, S = _oracle(c)
    check(y_host(Y), yref, S, out, f"ffn T={T} H={H} I={I} {xdt}->{out}")


@pytest.mark.parametrize("bn", [32, 64, 128, 192, 256])
@pytest.mark.parametrize("ks", [1, 2])
@pytest.mark.parametrize("pair", [1, 2])
def test_ffn_gateup_tile_options(bn, ks, pair):
    """Every token tile, K split and CTA-pair setting of the gate/up kernel,
    at I = 256 (four 64-row gate tiles) and I = 768 (twelve), ragged T."""
    for I in (256, 768):
        c = _case(9100 + bn + ks + I, 300, 512, I, "bf16")
        with _Opt(cq.CQ_OPT_TC_BN, bn), _Opt(cq.CQ_OPT_TC_KSPLIT, ks), _Opt(cq.CQ_OPT_TC_PAIR, pair):
            Y = _run(c, "f32")
        yref, S = _oracle(c)
        check(y_host(Y), yref, S, "f32", f"ffn bn={bn} ks={ks} pair={pair} I={I}")


def test_ffn_deterministic():
    c = _case(9200, 200, 512, 512)
    a = _run(c, "f32")
    b = _run(c, "f32")
    assert torch.equal(a, b)


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_ffn_denoiser_block_full_size(out):
    """The denoiser block's chain at 1024 target rows with its configured
    weights: gate/up [2 x 12288][3072] and down [3072][12288] (Q4), X bf16
    N(0, 0.5); every one of the 1024 x 3072 outputs against the f64 chain."""
    gu, dn = synth.c3()
    c = {"x": gu["x"], "x_dtype": "bf16", "guq": pack.pack_q4(gu["codes"]), "gus": gu["scales"],
         "dq": pack.pack_q4(dn["codes"]), "ds": dn["scales"], "T": 1024, "H": 3072, "I": 12288}
    Y = _run(c, out)
    yref, S = _oracle(c)
    check(y_host(Y), yref, S, out, f"ffn denoiser block {out}")
