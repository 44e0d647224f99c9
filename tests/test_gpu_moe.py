"""GPU parity of the routed MoE expert panels against the CPU oracle:
the routing layout bit-exact, the output within the acceptance bound."""
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


def _run(m, idx=None, w=None, out="f32", Y=None, expect=0):
    T, H, I, E = m["T"], m["H"], m["I"], m["E"]
    idx = m["idx"] if idx is None else idx
    w = m["w"] if w is None else w
    topk = idx.shape[1]
    guq = pack.pack_q4(m["gu_codes"])
    dq = pack.pack_q4(m["d_codes"])
    X = to_dev_x(m["x"], m["x_dtype"])
    if Y is None:
        Y = torch.empty(T, H, dtype=TORCH_DT[out], device=DEV)
    ws = torch.empty(cq.cq_moe_workspace_bytes(T, H, I, E, topk), dtype=torch.uint8, device=DEV)
    cq.cq_moe_panels(X, to_dev(np.ascontiguousarray(idx, np.int32)), to_dev(np.ascontiguousarray(w, np.float32)),
                     to_dev(guq), to_dev(m["gu_scales"]), to_dev(dq), to_dev(m["d_scales"]), Y, ws)
    st = cq.cq_get_device_error()
    assert st == expect, cq.STATUS[st]
    return Y, ws, guq, dq


def _oracle(m, guq, dq, idx=None, w=None):
    idx = m["idx"] if idx is None else idx
    w = m["w"] if w is None else w
    return oracle.moe(oracle.x_to_f64(m["x"], m["x_dtype"]), idx, w, guq, m["gu_scales"], dq, m["d_scales"],
                      m["E"], m["I"])


def _layout(ws, m, topk):
    P = m["T"] * topk
    perm = torch.empty(P, dtype=torch.int32, device=DEV)
    seg = torch.empty(m["E"] + 1, dtype=torch.int32, device=DEV)
    cq.cq_moe_layout(ws, m["T"], m["H"], m["I"], m["E"], topk, perm, seg)
    torch.cuda.synchronize()
    return perm.cpu().numpy(), seg.cpu().numpy()


def test_moe_pages_test_shape_uneven_loads():
    """The pages' MoE test layout ("oxinfer 0.0.5 src/metal.rs", tests
    module, mma_moe_matches_cpu): 8 experts, 75 tokens, top-2 with weights
    0.7 / 0.3, expert 5 unused, uneven loads (sizes raised to the shape rules)."""
    m = synth.moe_case(7, T=75, H=256, I=256, E=8, topk=2)
    idx = np.array([[[0, 1, 2, 3, 4, 6, 7][i % 7], [1, 7][i % 2]] for i in range(75)], np.int32)
    w = np.tile(np.array([0.7, 0.3], np.float32), (75, 1))
    for out in ("f32", "bf16"):
        Y, ws, guq, dq = _run(m, idx, w, out)
        yref, S = _oracle(m, guq, dq, idx, w)
        check(y_host(Y), yref, S, out, f"moe pages-shape {out}")
    perm, seg = _layout(ws, m, 2)
    operm, oseg = oracle.moe_layout(idx, 8)
    assert np.array_equal(perm, operm) and np.array_equal(seg, oseg)


@pytest.mark.parametrize("T,topk", [(1, 1), (5, 3), (40, 8)])
def test_moe_small_random(T, topk):
    m = synth.moe_case(20 + T, T=T, H=512, I=256, E=16, topk=topk)
    Y, ws, guq, dq = _run(m)
    yref, S = _oracle(m, guq, dq)
    check(y_host(Y), yref, S, "f32", f"moe T={T} topk={topk}")
    perm, seg = _layout(ws, m, topk)
    operm, oseg = oracle.moe_layout(m["idx"], 16)
    assert np.array_equal(perm, operm) and np.array_equal(seg, oseg)


def test_moe_hot_expert_many_pairs():
    """One expert receives more pairs than one column group holds (80 > 8),
    and repeated experts in a row count twice."""
    m = synth.moe_case(31, T=40, H=256, I=256, E=4, topk=2)
    idx = np.zeros((40, 2), np.int32)
    idx[::3, 1] = 2
    w = np.full((40, 2), 0.5, np.float32)
    Y, ws, guq, dq = _run(m, idx, w)
    yref, S = _oracle(m, guq, dq, idx, w)
    check(y_host(Y), yref, S, "f32", "moe hot expert")
    perm, seg = _layout(ws, m, 2)
    operm, oseg = oracle.moe_layout(idx, 4)
    assert np.array_equal(perm, operm) and np.array_equal(seg, oseg)


def test_moe_c4_full():
    """32 tokens, 128 experts, H=2048, I=768, top-8: every output compared."""
    m = synth.c4()
    for out in ("f32", "bf16"):
        Y, ws, guq, dq = _run(m, out=out)
        yref, S = _oracle(m, guq, dq)
        check(y_host(Y), yref, S, out, f"C4 {out}")
    perm, seg = _layout(ws, m, 8)
    operm, oseg = oracle.moe_layout(m["idx"], 128)
    assert np.array_equal(perm, operm) and np.array_equal(seg, oseg)


def test_moe_bad_index_reports_and_leaves_y():
    m = synth.moe_case(41, T=6, H=256, I=256, E=4, topk=2)
    idx = m["idx"].copy()
    idx[3, 1] = 4                                   # == E: out of range
    Y = torch.full((6, 256), 7.0, dtype=torch.float32, device=DEV)
    _run(m, idx=idx, Y=Y, expect=5)                 # CQ_ERR_INDEX
    assert torch.all(Y == 7.0)
    Y2, _, guq, dq = _run(m)                        # the next call is clean
    yref, S = _oracle(m, guq, dq)
    check(y_host(Y2), yref, S, "f32", "after bad index")


def test_moe_deterministic():
    m = synth.moe_case(42, T=32, H=512, I=256, E=16, topk=4)
    a = _run(m)[0]
    b = _run(m)[0]
    assert torch.equal(a, b)


def test_device_errors_are_per_stream():
    """A bad routing index on one stream sets that stream's error word only:
    a clean call on a second stream reports CQ_OK, the first stream reports
    CQ_ERR_INDEX once, and reading clears it."""
    m = synth.moe_case(43, T=6, H=256, I=256, E=4, topk=2)
    idx = m["idx"].copy()
    idx[2, 0] = -1
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    guq, dq = pack.pack_q4(m["gu_codes"]), pack.pack_q4(m["d_codes"])
    args = (to_dev_x(m["x"], "bf16"), to_dev(np.ascontiguousarray(idx, np.int32)), to_dev(m["w"]), to_dev(guq),
            to_dev(m["gu_scales"]), to_dev(dq), to_dev(m["d_scales"]))
    Y = torch.zeros(6, 256, dtype=torch.float32, device=DEV)
    ws = torch.empty(cq.cq_moe_workspace_bytes(6, 256, 256, 4, 2), dtype=torch.uint8, device=DEV)
    torch.cuda.synchronize()
    cq.cq_moe_panels(*args, Y, ws, stream=sa)
    case = synth.gemm_q4_case(44, 8, 512, 128)
    wq = pack.pack_q4(case["codes"])
    Yb = torch.empty(8, 128, dtype=torch.float32, device=DEV)
    wsb = torch.empty(cq.cq_gemm_q4_workspace_bytes(8, 512), dtype=torch.uint8, device=DEV)
    cq.cq_gemm_q4(to_dev_x(case["x"], "bf16"), to_dev(wq), to_dev(case["scales"]), Yb, wsb, stream=sb)
    assert cq.cq_get_device_error(sb) == 0
    assert cq.cq_get_device_error(sa) == 5                 # CQ_ERR_INDEX
    assert cq.cq_get_device_error(sa) == 0                 # cleared by the read
    yref, S = oracle.gemm_q4(wq, case["scales"], 128, 512, oracle.x_to_f64(case["x"], "bf16"))
    check(y_host(Yb), yref, S, "f32", "clean call on the other stream")


def test_moe_reused_workspace_of_any_contents():
    """The workspace starts as 0xFF bytes and serves three calls in a row with
    two routings: the down panels' row-block counters are reset by every call,
    so each result matches the oracle and the repeated call is bit-identical."""
    m = synth.moe_case(45, T=16, H=512, I=256, E=8, topk=4)
    T, H, I, E, topk = 16, 512, 256, 8, 4
    rng = np.random.default_rng(46)
    idx2 = np.stack([rng.permutation(E)[:topk] for _ in range(T)]).astype(np.int32)
    w2 = rng.uniform(0.1, 1.0, (T, topk)).astype(np.float32)
    guq, dq = pack.pack_q4(m["gu_codes"]), pack.pack_q4(m["d_codes"])
    X = to_dev_x(m["x"], "bf16")
    G = (to_dev(guq), to_dev(m["gu_scales"]), to_dev(dq), to_dev(m["d_scales"]))
    ws = torch.full((cq.cq_moe_workspace_bytes(T, H, I, E, topk),), 0xFF, dtype=torch.uint8, device=DEV)
    outs = []
    for idx, w in ((m["idx"], m["w"]), (idx2, w2), (m["idx"], m["w"])):
        Y = torch.full((T, H), float("nan"), dtype=torch.float32, device=DEV)
        cq.cq_moe_panels(X, to_dev(np.ascontiguousarray(idx, np.int32)), to_dev(np.ascontiguousarray(w)), *G, Y, ws)
        assert cq.cq_get_device_error() == 0
        yref, S = oracle.moe(oracle.x_to_f64(m["x"], "bf16"), idx, w, guq, m["gu_scales"], dq, m["d_scales"], E, I)
        check(y_host(Y), yref, S, "f32", "moe reused workspace")
        outs.append(Y)
    assert torch.equal(outs[0], outs[2])
