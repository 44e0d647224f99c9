"""GPU parity of the device routing (router logits -> top-k experts and
renormalised weights, the shared expert's sigmoid-gated slot) against the
CPU oracle: the expert indices bit-exact (both sides pick by comparing the
f32 logits), the weights (f32 exponentials on the device, f64 in the oracle)
within 8 f32 ulps;
then the whole routed MoE block with a shared expert (device routing, then
the expert panels with the shared expert stacked as expert E) against the
oracle's f64 chain."""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_weight_02_gb300 as cq
from block_quantized_weight_02_gb300 import pack, synth

from cqtest import DEV, check, to_dev, to_dev_x, y_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_dev):
    import __graft_entry__
    __graft_entry__.build()


def _route_dev(lg, topk, shared):
    T = lg.shape[0]
    slots = topk + (1 if shared else 0)
    idx = torch.full((T, slots), -7, dtype=torch.int32, device=DEV)
    w = torch.full((T, slots), float("nan"), dtype=torch.float32, device=DEV)
    cq.cq_moe_route(to_dev(np.ascontiguousarray(lg, np.float32)), topk, idx, w, shared=shared)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T,E,topk", [(1, 8, 1), (32, 128, 8), (77, 1024, 64), (300, 40, 33), (5, 64, 64)])
@pytest.mark.parametrize("shared", [False, True])
def test_route_matches_oracle(T, E, topk, shared):
    rng = np.random.default_rng(9600 + T + E + topk)
    lg = rng.standard_normal((T, E + (1 if shared else 0))).astype(np.float32)
    lg[0, : E // 2] = 0.25                       # a run of equal logits: ties go to the lower index
    idx, w = _route_dev(lg, topk, shared)
    oidx, ow = oracle.route(lg, topk, shared)
    assert np.array_equal(idx, oidx)
    assert np.all(np.abs(w - ow) <= 8 * np.spacing(np.abs(ow)))


def test_route_heavy_ties():
    rng = np.random.default_rng(9700)
    lg = (rng.integers(-2, 3, (64, 256)) * 0.5).astype(np.float32)
    idx, w = _route_dev(lg, 16, False)
    oidx, ow = oracle.route(lg, 16)
    assert np.array_equal(idx, oidx)
    assert np.all(np.abs(w - ow) <= 8 * np.spacing(np.abs(ow)))


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_moe_block_with_device_routing_and_shared_expert(out):
    """32 tokens, 16 routed experts + 1 shared (stacked as expert 16), top-4:
    routing on the device from the logits, then the panels; against the
    oracle's routing and f64 chain, the layout bit-exact."""
    T, H, I, E, topk = 32, 512, 256, 16, 4
    m = synth.moe_case(9800, T=T, H=H, I=I, E=E + 1, topk=topk)
    rng = np.random.default_rng(9801)
    lg = rng.standard_normal((T, E + 1)).astype(np.float32)
    idx_d = torch.empty(T, topk + 1, dtype=torch.int32, device=DEV)
    w_d = torch.empty(T, topk + 1, dtype=torch.float32, device=DEV)
    cq.cq_moe_route(to_dev(lg), topk, idx_d, w_d, shared=True)
    guq, dq = pack.pack_q4(m["gu_codes"]), pack.pack_q4(m["d_codes"])
    Y = torch.full((T, H), float("nan"), dtype=torch.float32 if out == "f32" else torch.bfloat16, device=DEV)
    ws = torch.empty(cq.cq_moe_workspace_bytes(T, H, I, E + 1, topk + 1), dtype=torch.uint8, device=DEV)
    cq.cq_moe_panels(to_dev_x(m["x"], "bf16"), idx_d, w_d, to_dev(guq), to_dev(m["gu_scales"]), to_dev(dq),
                     to_dev(m["d_scales"]), Y, ws)
    assert cq.cq_get_device_error() == 0
    oidx, ow = oracle.route(lg, topk, shared=True)
    assert np.array_equal(idx_d.cpu().numpy(), oidx)
    yref, S = oracle.moe(oracle.x_to_f64(m["x"], "bf16"), oidx, ow, guq, m["gu_scales"], dq, m["d_scales"], E + 1, I)
    check(y_host(Y), yref, S, out, f"moe with device routing and a shared expert ({out})")
    perm = torch.empty(T * (topk + 1), dtype=torch.int32, device=DEV)
    seg = torch.empty(E + 2, dtype=torch.int32, device=DEV)
    cq.cq_moe_layout(ws, T, H, I, E + 1, topk + 1, perm, seg)
    torch.cuda.synchronize()
    operm, oseg = oracle.moe_layout(oidx, E + 1)
    assert np.array_equal(perm.cpu().numpy(), operm) and np.array_equal(seg.cpu().numpy(), oseg)
