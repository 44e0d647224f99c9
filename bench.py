"""Benchmark of the quantized-weight GEMM path on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
                [--no-per-config] [--no-cpu-baseline] [--eager] [--traffic-pass]

Default workload "denoiser_block" (the largest configuration): one step = the
two Q4 GEMMs of the denoiser block at 1024 target rows, gate/up (T=1024,
K=3072, N=2x12288) then down (T=1024, K=12288, N=3072), bf16 outputs.  The
metric is dequant-GEMM TFLOP/s (2*T*N*K per call, all calls of all ranks over
the max-over-ranks time); weight GB/s and the roofline fraction of the
dominant call ride along in the same JSON line.

Beside it, "per_config" times every call of the other configurations alone,
each in a back-to-back chain of its own over input sets larger than L2: the
smallest Q4 case, the prefill projection (Q4 and Q8-row, f32 and bf16), the
MoE expert panels and the decode-to-prefill sweep (Q4 and Q8-row at
T = 1, 8, 32, 128, 512, 2048).  Each entry gives microseconds per call,
TFLOP/s, weight GB/s, the fractions of the measured tensor and HBM peaks, the
bound (whichever roofline is lower for the call's arithmetic intensity) and
the DRAM traffic per call from the committed ncu summary
(profiles/traffic_per_call.md), or null once the kernel sources have changed
since it was taken.

Other workloads for the headline: smallest_q4, prefill_projection_4096,
moe_panels, sweep_q4_T<T>, sweep_q8_T<T>.

Under torchrun (N > 1) every rank runs its own copy of the workload
(independent problems, no collective on the data path): weak scaling.
--impl reference times the CPU oracle on a bounded sample of the same
workload (rank 0 only).  --traffic-pass runs every call of every
configuration once, after one warm-up call each, and exits (the command the
ncu traffic summary is taken over).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 2**20


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# workloads: inputs on the device, a list of calls per step
# ---------------------------------------------------------------------------

class Call:
    """One C-ABI call with its algorithmic work and the buffers it reads and writes.
    Its kernel launches are counted by the library (cq_last_launches) when the call
    runs through run_counted(); `counter` replaces that for a step of several
    library calls (it runs them and returns their launches)."""

    def __init__(self, name, fn, flops, weight_bytes, other_bytes, h2d=(), d2h=(), counter=None):
        self.name, self.fn, self.flops = name, fn, flops
        self.weight_bytes, self.other_bytes = weight_bytes, other_bytes
        self.launches = None
        self.h2d, self.d2h = list(h2d), list(d2h)
        self.counter = counter

    def run_counted(self):
        import block_quantized_weight_02_gb300 as cq
        if self.counter is not None:
            self.launches = int(self.counter())
        else:
            self.fn()
            self.launches = int(cq.cq_last_launches())
        return self.launches


def _dev_x(x_bits, dtype, dev):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16))
    return t.view(torch.bfloat16 if dtype == "bf16" else torch.float16).to(dev)


def _u16(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)


def _q4_calls(cq, case, outs, dev, tag):
    import torch
    from block_quantized_weight_02_gb300 import pack
    T, K, N = case["T"], case["K"], case["N"]
    X = _dev_x(case["x"], case["x_dtype"], dev)
    Wq = torch.from_numpy(pack.pack_q4(case["codes"])).to(dev)
    Ws = _u16(case["scales"], dev)
    ws = torch.empty(cq.cq_gemm_q4_workspace_bytes(T, K), dtype=torch.uint8, device=dev)
    calls = []
    wbytes = N * K // 2 + N * K // 32 * 2
    for out in outs:
        Y = torch.empty(T, N, dtype=torch.float32 if out == "f32" else torch.bfloat16, device=dev)
        calls.append(Call(f"{tag} q4->{out}", (lambda X=X, Wq=Wq, Ws=Ws, Y=Y, ws=ws: cq.cq_gemm_q4(X, Wq, Ws, Y, ws)),
                          2.0 * T * N * K, wbytes, X.numel() * 2 + Y.numel() * Y.element_size(),
                          h2d=[X], d2h=[Y]))
    return calls


def _q8_calls(cq, case, outs, dev, tag):
    import torch
    T, K, N = case["T"], case["K"], case["N"]
    X = _dev_x(case["x"], case["x_dtype"], dev)
    Wq = torch.from_numpy(case["q"]).to(dev)
    rs = torch.from_numpy(case["rs"]).to(dev)
    calls = []
    for out in outs:
        Y = torch.empty(T, N, dtype=torch.float32 if out == "f32" else torch.bfloat16, device=dev)
        calls.append(Call(f"{tag} q8row->{out}", (lambda X=X, Wq=Wq, rs=rs, Y=Y: cq.cq_gemm_q8row(X, Wq, rs, Y)),
                          2.0 * T * N * K, N * K + 4 * N, X.numel() * 2 + Y.numel() * Y.element_size(),
                          h2d=[X], d2h=[Y]))
    return calls


def _moe_calls(cq, m, dev):
    import torch
    from block_quantized_weight_02_gb300 import pack
    T, H, I, E, topk = m["T"], m["H"], m["I"], m["E"], m["topk"]
    X = _dev_x(m["x"], m["x_dtype"], dev)
    idx = torch.from_numpy(m["idx"]).to(dev)
    w = torch.from_numpy(m["w"]).to(dev)
    guq = torch.from_numpy(pack.pack_q4(m["gu_codes"])).to(dev)
    gus = _u16(m["gu_scales"], dev)
    dq = torch.from_numpy(pack.pack_q4(m["d_codes"])).to(dev)
    ds = _u16(m["d_scales"], dev)
    Y = torch.empty(T, H, dtype=torch.float32, device=dev)
    ws = torch.empty(cq.cq_moe_workspace_bytes(T, H, I, E, topk), dtype=torch.uint8, device=dev)
    touched = len(np.unique(m["idx"]))
    per_expert = (2 * I * H + H * I) * 9 // 16
    flops = T * topk * (2.0 * H * 2 * I + 2.0 * I * H)
    return [Call("moe panels", lambda: cq.cq_moe_panels(X, idx, w, guq, gus, dq, ds, Y, ws), flops,
                 touched * per_expert, X.numel() * 2 + Y.numel() * 4 + idx.numel() * 8,
                 h2d=[X, idx, w], d2h=[Y])], touched


def _ffn_calls(cq, gu, dn, dev):
    """The denoiser block as one chained call: gate/up GEMM with SwiGLU in its
    epilogue, then the down GEMM, on the configured weights and the gate/up X."""
    import torch
    from block_quantized_weight_02_gb300 import pack
    T, H, I = gu["T"], gu["K"], gu["N"] // 2
    X = _dev_x(gu["x"], gu["x_dtype"], dev)
    guq = torch.from_numpy(pack.pack_q4(gu["codes"])).to(dev)
    gus = _u16(gu["scales"], dev)
    dq = torch.from_numpy(pack.pack_q4(dn["codes"])).to(dev)
    ds = _u16(dn["scales"], dev)
    Y = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(cq.cq_ffn_q4_workspace_bytes(T, H, I), dtype=torch.uint8, device=dev)
    wbytes = (2 * I * H + H * I) * 9 // 16
    return [Call("ffn chain q4->bf16", lambda: cq.cq_ffn_q4(X, guq, gus, dq, ds, Y, ws),
                 2.0 * T * (2 * I * H + H * I), wbytes, X.numel() * 2 + Y.numel() * 2,
                 h2d=[X], d2h=[Y])]


def _moe_routed_calls(cq, m, dev):
    """The MoE block from its router logits: routing on the device (softmax,
    top-8, renormalised weights), then the expert panels, as one step."""
    import torch
    from block_quantized_weight_02_gb300 import pack
    T, H, I, E, topk = m["T"], m["H"], m["I"], m["E"], m["topk"]
    X = _dev_x(m["x"], m["x_dtype"], dev)
    lg = torch.from_numpy(np.ascontiguousarray(m["logits"], np.float32)).to(dev)
    idx = torch.empty(T, topk, dtype=torch.int32, device=dev)
    w = torch.empty(T, topk, dtype=torch.float32, device=dev)
    guq = torch.from_numpy(pack.pack_q4(m["gu_codes"])).to(dev)
    gus = _u16(m["gu_scales"], dev)
    dq = torch.from_numpy(pack.pack_q4(m["d_codes"])).to(dev)
    ds = _u16(m["d_scales"], dev)
    Y = torch.empty(T, H, dtype=torch.float32, device=dev)
    ws = torch.empty(cq.cq_moe_workspace_bytes(T, H, I, E, topk), dtype=torch.uint8, device=dev)
    touched = len(np.unique(m["idx"]))
    per_expert = (2 * I * H + H * I) * 9 // 16
    flops = T * topk * (2.0 * H * 2 * I + 2.0 * I * H)

    def fn():
        cq.cq_moe_route(lg, topk, idx, w)
        cq.cq_moe_panels(X, idx, w, guq, gus, dq, ds, Y, ws)

    def counter():
        cq.cq_moe_route(lg, topk, idx, w)
        n = cq.cq_last_launches()
        cq.cq_moe_panels(X, idx, w, guq, gus, dq, ds, Y, ws)
        return n + cq.cq_last_launches()
    return [Call("route + moe panels", fn, flops, touched * per_expert, X.numel() * 2 + Y.numel() * 4 + lg.numel() * 4,
                 h2d=[X, lg], d2h=[Y], counter=counter)], touched


_HOST_CACHE = {}


def _host_arrays(key, fn):
    """Seeded host inputs built once per process (the rotating sets copy them to the device)."""
    if key not in _HOST_CACHE:
        _HOST_CACHE[key] = fn()
    return _HOST_CACHE[key]


def _batched_calls(cq, dev):
    """z-batched Q4: three weights of one shape sharing one X (a qkv projection),
    T=512, K=N=4096 each, outputs side by side in Y[512][3*4096] bf16."""
    import torch
    from block_quantized_weight_02_gb300 import pack, synth
    T, K, N, z = 512, 4096, 4096, 3

    def draw():
        rng = np.random.default_rng(11)
        x = synth.draw_x(rng, T, K, 1.0, "bf16")
        ws = [synth.draw_q4(rng, N, K) for _ in range(z)]
        return x, [(pack.pack_q4(c), np.ascontiguousarray(sc).view(np.uint16)) for c, sc in ws]
    x, packed = _host_arrays("batched", draw)
    X = _dev_x(x, "bf16", dev)
    jobs = [(torch.from_numpy(q).to(dev), _u16(sc, dev), 0, j * N) for j, (q, sc) in enumerate(packed)]
    Y = torch.empty(T, z * N, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(cq.cq_gemm_q4_batched_workspace_bytes(T, K, z), dtype=torch.uint8, device=dev)
    wbytes = z * (N * K // 2 + N * K // 32 * 2)
    return [Call("qkv z=3 q4->bf16", lambda: cq.cq_gemm_q4_batched(X, K, jobs, N, Y, ws), 2.0 * T * z * N * K, wbytes,
                 X.numel() * 2 + Y.numel() * 2, h2d=[X], d2h=[Y])]


def _format_calls(cq, dev):
    """The format variants at K=N=4096, bf16 out, each at T=8 (weight streaming) and
    T=512 (tcgen05): Q8 per 32-k block, affine Q4 (one bf16 offset per 2 blocks) and
    q8_2f (int8 times a column field, f32 row scale)."""
    import torch
    from block_quantized_weight_02_gb300 import pack, synth
    K, N, gk = 4096, 4096, 2

    def draw():
        rng = np.random.default_rng(12)
        q8 = rng.integers(-127, 128, (N, K)).astype(np.int8)
        s8b = (rng.uniform(1e-3, 1e-2, (N, K // 32)) * np.where(rng.random((N, K // 32)) < 0.5, -1, 1)).astype(np.float32)
        codes, sc = synth.draw_q4(rng, N, K, signed=True)
        off = synth.f32_to_bf16_bits(rng.uniform(-0.15, 0.15, (N, K // 32 // gk)).astype(np.float32))
        rs = rng.uniform(1e-3, 1e-2, N).astype(np.float32)
        col = rng.uniform(0.25, 4.0, K).astype(np.float16).astype(np.float32)
        xs = {T: synth.draw_x(rng, T, K, 1.0, "bf16") for T in (8, 512)}
        return q8, s8b, pack.pack_q4(codes), np.ascontiguousarray(sc).view(np.uint16), off, rs, col, xs
    q8, s8b, q4p, sc, off, rs, col, xs = _host_arrays("formats", draw)
    Q8 = torch.from_numpy(q8).to(dev)
    S8B = torch.from_numpy(s8b).to(dev)
    Q4 = torch.from_numpy(q4p).to(dev)
    SC = _u16(sc, dev)
    OFF = _u16(off, dev)
    RS = torch.from_numpy(rs).to(dev)
    COL = torch.from_numpy(col).to(dev)
    calls = []
    for T in (8, 512):
        X = _dev_x(xs[T], "bf16", dev)
        fl = 2.0 * T * N * K
        xb = X.numel() * 2 + T * N * 2
        Yb = torch.empty(T, N, dtype=torch.bfloat16, device=dev)
        wsb = torch.empty(cq.cq_gemm_q8b_workspace_bytes(T, K), dtype=torch.uint8, device=dev)
        calls.append(Call(f"T{T} q8b->bf16", (lambda X=X, Y=Yb, ws=wsb: cq.cq_gemm_q8b(X, Q8, S8B, Y, ws)), fl,
                          N * K + N * K // 32 * 4, xb, h2d=[X], d2h=[Yb]))
        Ya = torch.empty(T, N, dtype=torch.bfloat16, device=dev)
        wsa = torch.empty(cq.cq_gemm_q4a_workspace_bytes(T, K, N, gk), dtype=torch.uint8, device=dev)
        calls.append(Call(f"T{T} q4a->bf16", (lambda X=X, Y=Ya, ws=wsa: cq.cq_gemm_q4a(X, Q4, SC, OFF, gk, Y, ws)), fl,
                          N * K // 2 + N * K // 32 * 2 + N * K // 32 // gk * 2, xb, h2d=[X], d2h=[Ya]))
        Yf = torch.empty(T, N, dtype=torch.bfloat16, device=dev)
        wsf = torch.empty(cq.cq_gemm_q8_2f_workspace_bytes(T, K), dtype=torch.uint8, device=dev)
        calls.append(Call(f"T{T} q8_2f->bf16", (lambda X=X, Y=Yf, ws=wsf: cq.cq_gemm_q8_2f(X, Q8, RS, COL, Y, ws)), fl,
                          N * K + 4 * N + 4 * K, xb, h2d=[X], d2h=[Yf]))
    return calls


def _dtype_of(name, info):
    """The arithmetic each call of the workload runs in: the tcgen05 path (T > 32)
    multiplies guarded fp16 activations by fp16 weights; the weight-streaming path
    (T <= 32) multiplies the activations as given (bf16 here, fp16 for the smallest
    case) by the exact nibble - 8 and scales each 32-k block in f32; Q8-row is
    bf16 x bf16 (int8 exact); all accumulate in f32."""
    if name.startswith("moe"):
        return "q4:fp16xfp16->f32"
    if name == "smallest_q4":
        return "q4:fp16xfp16->f32"
    if name == "formats_4096":
        return ("T8: q8b/q4a bf16xbf16->f32, q8_2f fp16xfp16->f32; "
                "T512: q8b/q8_2f/q4a fp16xfp16->f32")
    T = info.get("T", 0)
    q4 = "q4:bf16xbf16->f32" if T <= 32 else "q4:fp16xfp16->f32"
    if name == "prefill_projection_4096":
        return q4 + ", q8row:bf16xbf16->f32"

    if name.startswith("sweep_q8"):
        return "q8row:bf16xbf16->f32"
    return q4


def build_workload(name, dev, max_sets=16):
    import block_quantized_weight_02_gb300 as cq
    from block_quantized_weight_02_gb300 import synth
    info = {}
    if name == "prefill_projection_4096":
        c4, c8 = synth.c2_q4(), synth.c2_q8()
        make = lambda: _q4_calls(cq, c4, ["f32", "bf16"], dev, "T512") + _q8_calls(cq, c8, ["f32", "bf16"], dev, "T512")
        info = {"T": 512, "K": 4096, "N": 4096, "formats": ["q4", "q8row"], "outputs": ["f32", "bf16"]}
    elif name == "smallest_q4":
        c = synth.c1()
        make = lambda: _q4_calls(cq, c, ["f32"], dev, "T16")
        info = {"T": 16, "K": 512, "N": 256, "formats": ["q4"], "outputs": ["f32"]}
    elif name == "denoiser_block":
        gu, dn = synth.c3()
        make = lambda: _q4_calls(cq, gu, ["bf16"], dev, "gate/up") + _q4_calls(cq, dn, ["bf16"], dev, "down")
        info = {"T": 1024, "gate_up": [3072, 24576], "down": [12288, 3072], "formats": ["q4"], "outputs": ["bf16"]}
    elif name == "denoiser_ffn_chain":
        gu, dn = synth.c3()
        make = lambda: _ffn_calls(cq, gu, dn, dev)
        info = {"T": 1024, "H": 3072, "I": 12288, "formats": ["q4"], "outputs": ["bf16"],
                "chain": "gate/up + SwiGLU epilogue -> guard -> down"}
    elif name == "moe_routed_from_logits":
        m = synth.c4()
        calls, touched = _moe_routed_calls(cq, m, dev)
        info = {"T": 32, "H": 2048, "I": 768, "E": 128, "topk": 8, "touched_experts": touched, "outputs": ["f32"],
                "routing": "on the device from the router logits"}
        return (lambda: [calls]), info, 1
    elif name == "moe_panels":
        m = synth.c4()
        calls, touched = _moe_calls(cq, m, dev)
        info = {"T": 32, "H": 2048, "I": 768, "E": 128, "topk": 8, "touched_experts": touched, "outputs": ["f32"]}
        return (lambda: [calls]), info, 1
    elif name == "batched_qkv_4096":
        make = lambda: _batched_calls(cq, dev)
        info = {"T": 512, "K": 4096, "N": 4096, "z": 3, "shared_x": True, "formats": ["q4"], "outputs": ["bf16"]}
    elif name == "formats_4096":
        make = lambda: _format_calls(cq, dev)
        info = {"T": [8, 512], "K": 4096, "N": 4096, "formats": ["q8b", "q4a", "q8_2f"], "outputs": ["bf16"]}
    elif name.startswith("sweep_q4_T") or name.startswith("sweep_q8_T"):
        T = int(name.split("_T")[1])
        if "q4" in name:
            c = synth.c5_q4(T)
            make = lambda: _q4_calls(cq, c, ["bf16"], dev, f"T{T}")
        else:
            c = synth.c5_q8(T)
            make = lambda: _q8_calls(cq, c, ["bf16"], dev, f"T{T}")
        info = {"T": T, "K": 8192, "N": 8192, "outputs": ["bf16"]}
    else:
        raise SystemExit(f"unknown workload {name}")
    one = make()
    set_bytes = sum(c.weight_bytes + c.other_bytes for c in one)
    sets = max(1, min(max_sets, -(-3 * L2_BYTES // max(set_bytes, 1))))
    rot = [one] + [make() for _ in range(sets - 1)]
    return (lambda i=[0]: rot), info, sets


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class Clocks:
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.path = index, None, None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 8:
                rows.append(f)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def max_over_ranks(value: float, world: int) -> float:
    """The slowest rank's number (timing only; no data-path collective)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_step: float, world: int, ms_per_step_max: float) -> float:
    """Weak scaling: every rank processes `units_per_step`; the job's rate is
    all ranks' units over the slowest rank's time."""
    return units_per_step * world / (ms_per_step_max * 1e-3)


PER_CONFIG = (["smallest_q4", "prefill_projection_4096", "denoiser_ffn_chain", "moe_panels", "moe_routed_from_logits",
               "batched_qkv_4096", "formats_4096"]
              + [f"sweep_{f}_T{t}" for f in ("q4", "q8") for t in (1, 8, 32, 128, 512, 2048)])

TRAFFIC_MD = os.path.join(ROOT, "profiles", "traffic_per_call.md")


def kernel_sources_hash() -> str:
    """Hash of the library's kernel sources and header: the DRAM traffic taken
    with ncu belongs to the kernels built from exactly these files."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_quantized_weight_02_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            h.update(f.encode())
            h.update(open(os.path.join(csrc, f), "rb").read())
    h.update(open(os.path.join(ROOT, "include", "cq.h"), "rb").read())
    return h.hexdigest()[:16]


def load_traffic(path=TRAFFIC_MD):
    """{(workload, call): DRAM bytes per call} from the committed ncu summary
    (rows `| workload | call | launches | DRAM bytes per call | ...`), empty when
    the summary was taken on other kernel sources."""
    if not os.path.exists(path):
        return {}
    txt = open(path).read()
    import re
    m = re.search(r"kernel sources `([0-9a-f]{16})`", txt)
    if not m or m.group(1) != kernel_sources_hash():
        return {}
    out = {}
    for line in txt.splitlines():
        cells = [c.strip().strip("`") for c in line.strip().strip("|").split("|")]
        if len(cells) >= 4 and (cells[0] in PER_CONFIG or cells[0] == "denoiser_block"):
            try:
                out[(cells[0], cells[1])] = int(cells[3].replace(",", ""))
            except ValueError:
                pass
    return out


def roofline_entry(call, ms, peaks, traffic):
    """Throughput of one call and its fractions of the measured peaks.  The
    bound is the roofline the call's arithmetic intensity (FLOPs over its
    algorithmic bytes: weights + activations + outputs) puts it under."""
    s = ms * 1e-3
    alg = call.weight_bytes + call.other_bytes
    tf = call.flops / s / 1e12
    gbs = alg / s / 1e9
    ft, fh = tf / peaks["bf16_tflops"], gbs / peaks["hbm_gbs"]
    tensor = call.flops / max(alg, 1) > peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    return {"us": round(ms * 1e3, 3), "tflops": round(tf, 2), "weight_gbs": round(call.weight_bytes / s / 1e9, 1),
            "bytes_gbs": round(gbs, 1), "bound": "tensor" if tensor else "hbm",
            "frac": round(ft if tensor else fh, 4), "frac_tensor": round(ft, 4), "frac_hbm": round(fh, 4),
            "algorithmic_bytes": int(alg), "traffic": traffic, "launches": call.launches}


def time_calls(rot, sets, reps, stream, use_graph):
    """Average duration (ms) of each call of the step alone: the call repeated
    back to back over the rotating input sets, captured in a CUDA graph and
    replayed once untimed, then timed with CUDA events on the launching stream."""
    import torch
    out = []
    for j in range(len(rot[0])):
        n = rot[0][j].run_counted()   # one more untimed call: its kernel launches, as the library counts them
        torch.cuda.synchronize()
        for calls in rot:
            calls[j].launches = n
        g = None
        if use_graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for i in range(reps):
                    rot[i % sets][j].fn()
            g.replay()
            torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        if g is not None:
            g.replay()
        else:
            for i in range(reps):
                rot[i % sets][j].fn()
        b.record(stream)
        torch.cuda.synchronize()
        out.append(a.elapsed_time(b) / reps)
        del g
    return out


def traffic_pass(args, dev):
    """Every call of every configuration once after one warm-up call each, one
    input set, nothing timed: the launches an ncu DRAM-traffic capture reads.
    Prints the launch order (workload, call, launches) to stdout."""
    import torch
    import block_quantized_weight_02_gb300 as cq
    names = ["denoiser_block"] + PER_CONFIG if args.configs == "all" else args.configs.split(",")
    for name in names:
        rot_fn, info, sets = build_workload(name, dev, max_sets=1)
        calls = rot_fn()[0]
        for c in calls:
            c.fn()
            torch.cuda.synchronize()
            c.run_counted()
            torch.cuda.synchronize()
            print(f"traffic-pass\t{name}\t{c.name}\t{c.launches}", flush=True)
        if cq.cq_get_device_error() != 0:
            raise SystemExit(f"device error in {name}")
        del calls, rot_fn
        torch.cuda.empty_cache()


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import __graft_entry__
    __graft_entry__.build()
    import block_quantized_weight_02_gb300 as cq

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cq.cq_set_option(cq.CQ_OPT_STREAM_KERNEL, args.stream_kernel)
    if args.traffic_pass:
        traffic_pass(args, dev)
        return
    peaks = _peaks()
    traffic = load_traffic()
    rot_fn, info, sets = build_workload(args.workload, dev)
    rot = rot_fn()
    stream = torch.cuda.current_stream()

    def step(i):
        for c in rot[i % sets]:
            c.fn()

    def barrier():
        if world > 1:
            dist.barrier()

    # Clocks are sampled from the warm-up to the end of the per-call timings
    # (the K timed steps alone last milliseconds, shorter than a sample).
    clocks = Clocks(local_rank)
    clocks.start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if cq.cq_get_device_error() != 0:
        raise SystemExit("device error during warm-up")

    # The timed region: K steps of the workload's calls, back to back on one
    # stream.  By default it is captured once into a CUDA graph and replayed,
    # so host-side launch overhead does not leave the GPU idle between the
    # short calls and consecutive kernels overlap through their programmatic
    # dependencies; --eager times direct calls instead.
    timing = "eager"
    graph = None
    if not args.eager:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for i in range(args.steps):
                    for c in rot[i % sets]:
                        c.fn()
            timing = "cuda-graph replay"
        except Exception as exc:
            print(f"bench: graph capture unavailable ({exc!r}); timing direct calls", file=sys.stderr)
            graph = None
            torch.cuda.synchronize()
            cq.cq_get_device_error()
    if graph is not None:
        graph.replay()                    # one untimed replay
        torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            for c in rot[i % sets]:
                c.fn()
    t1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = t0.elapsed_time(t1)
    if cq.cq_get_device_error() != 0:
        raise SystemExit("device error during the timed region")
    ms_max = max_over_ranks(ms, world)

    # Per-call duration (for the roofline of the dominant call).
    reps = max(3, min(args.steps, 50))
    per_call_ms = time_calls(rot, sets, reps, stream, graph is not None)
    if cq.cq_get_device_error() != 0:
        raise SystemExit("device error while timing the calls")

    calls = rot[0]
    flops_step = sum(c.flops for c in calls)
    wbytes_step = sum(c.weight_bytes for c in calls)
    ms_step = ms_max / args.steps
    tflops = whole_job_rate(flops_step, world, ms_step) / 1e12
    wgbs = whole_job_rate(wbytes_step, world, ms_step) / 1e9

    # e2e: host buffers (pinned), every step the H2D copy of each call's inputs, the calls and
    # the D2H copy of their outputs.  With two or more input sets the copies run on their own
    # streams, so step i + 1's inputs and step i - 1's outputs move while step i computes
    # (each set's buffers are reused only after its previous step's copies are done).
    nb = min(sets, 3)
    host_in = [[[torch.empty_like(t, device="cpu").pin_memory() for t in c.h2d] for c in rot[b]] for b in range(nb)]
    host_out = [[[torch.empty_like(t, device="cpu").pin_memory() for t in c.d2h] for c in rot[b]] for b in range(nb)]
    for b in range(nb):
        for j, c in enumerate(rot[b]):
            for h, d in zip(host_in[b][j], c.h2d):
                h.copy_(d.cpu())
    h2d_b = sum(t.numel() * t.element_size() for c in calls for t in c.h2d)
    d2h_b = sum(t.numel() * t.element_size() for c in calls for t in c.d2h)
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(nb)]
    done = [torch.cuda.Event() for _ in range(nb)]
    out_done = [torch.cuda.Event() for _ in range(nb)]

    def e2e_run(nsteps, start_event=None):
        for i in range(nsteps):
            b = i % nb
            with torch.cuda.stream(h2d_s):
                if i == 0 and start_event is not None:
                    h2d_s.wait_event(start_event)
                if i >= nb:
                    h2d_s.wait_event(done[b])          # step i - nb has read set b's inputs
                for j, c in enumerate(rot[b]):
                    for h, d in zip(host_in[b][j], c.h2d):
                        d.copy_(h, non_blocking=True)
                in_ready[b].record(h2d_s)
            stream.wait_event(in_ready[b])
            if i >= nb:
                stream.wait_event(out_done[b])         # step i - nb's outputs have left set b
            for c in rot[b]:
                c.fn()
            done[b].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(done[b])
                for j, c in enumerate(rot[b]):
                    for h, d in zip(host_out[b][j], c.d2h):
                        h.copy_(d, non_blocking=True)
                out_done[b].record(d2h_s)
        stream.wait_event(out_done[(nsteps - 1) % nb])

    e2e_run(max(nb, args.warmup))
    torch.cuda.synchronize()
    e_steps = max(3, min(args.steps, 50))
    barrier()
    torch.cuda.synchronize()
    a, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    e2e_run(e_steps, a)
    b_ev.record(stream)
    torch.cuda.synchronize()
    e_ms = max_over_ranks(a.elapsed_time(b_ev) / e_steps, world)
    e2e_val = whole_job_rate(flops_step, world, e_ms) / 1e12

    # roofline of the dominant call (largest share of the step)
    j = int(np.argmax(per_call_ms))
    dom = calls[j]
    ent = roofline_entry(dom, per_call_ms[j], peaks, traffic.get((args.workload, dom.name)))
    roof = {"bound": ent["bound"], "achieved": ent["tflops"] if ent["bound"] == "tensor" else ent["bytes_gbs"],
            "peak": peaks["bf16_tflops"] if ent["bound"] == "tensor" else peaks["hbm_gbs"],
            "unit": "TFLOP/s" if ent["bound"] == "tensor" else "GB/s", "frac": ent["frac"],
            "traffic": ent["traffic"], "algorithmic_bytes": ent["algorithmic_bytes"], "kernel": dom.name,
            "launch_ms": round(per_call_ms[j], 5), "peak_source": peaks["source"],
            "launches_in_call": dom.launches}

    # every call of the other configurations, each alone in its own chain
    per_config = {args.workload: {c.name: roofline_entry(c, t, peaks, traffic.get((args.workload, c.name)))
                                  for c, t in zip(calls, per_call_ms)}}
    if not args.no_per_config:
        del rot, rot_fn, graph
        torch.cuda.empty_cache()
        for name in PER_CONFIG:
            if name == args.workload:
                continue
            r_fn, _, n_sets = build_workload(name, dev)
            r = r_fn()
            r[0][0].fn()                  # warm-up
            torch.cuda.synchronize()
            t_ms = time_calls(r, n_sets, 20 if name.endswith("T2048") else 50, stream, not args.eager)
            if cq.cq_get_device_error() != 0:
                raise SystemExit(f"device error while timing {name}")
            per_config[name] = {c.name: roofline_entry(c, t, peaks, traffic.get((name, c.name)))
                                for c, t in zip(r[0], t_ms)}
            del r, r_fn
            torch.cuda.empty_cache()
    clk = clocks.stop()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload)

    line = {
        "metric": "dequant-GEMM TFLOP/s (weight GB/s and roofline fraction alongside)",
        "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": _dtype_of(args.workload, info), "data": "synthetic (seeded)",
        "config": {"workload": args.workload, **info, "parallelism": f"replicas x{world}",
                   "timing": timing, **({"stream_kernel": args.stream_kernel} if args.stream_kernel else {}),
                   "l2": f"rotating {sets} input sets ({sets * sum(c.weight_bytes + c.other_bytes for c in calls) / 2**20:.0f} MiB) > L2"},
        "weight_gbs": round(wgbs, 1),
        "per_call_ms": {c.name: round(t, 5) for c, t in zip(calls, per_call_ms)},
        "roofline": roof,
        "e2e": {"value": round(e2e_val, 3), "unit": "TFLOP/s", "copies": f"own streams, {nb} buffer set(s)",
                "h2d_bytes_per_step": h2d_b,
                "d2h_bytes_per_step": d2h_b},
        "gpu_launches": sum(c.launches for c in calls) * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
        "per_config": per_config,
        "peaks": {"tensor_tflops": peaks["bf16_tflops"], "hbm_gbs": peaks["hbm_gbs"], "source": peaks["source"]},
        "traffic_source": "profiles/traffic_per_call.md" if traffic else None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# CPU oracle (the reference arm and the cpu_baseline object)
# ---------------------------------------------------------------------------

def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _oracle_sample(workload):
    """(make(rows) -> (fn, flops, description), max_rows): the oracle on the
    first `rows` activation rows (tokens) of the workload, full N and K."""
    import oracle
    from block_quantized_weight_02_gb300 import synth
    oracle.build()
    if workload == "prefill_projection_4096":
        c4, c8 = synth.c2_q4(), synth.c2_q8()
        wq = oracle.pack_q4(c4["codes"])

        def make(rows):
            X4 = oracle.x_to_f64(c4["x"][:rows], "bf16")
            X8 = oracle.x_to_f64(c8["x"][:rows], "bf16")

            def fn():
                oracle.gemm_q4(wq, c4["scales"], 4096, 4096, X4)
                oracle.gemm_q8row(c8["q"], c8["rs"], X8)
            return fn, 2 * 2.0 * rows * 4096 * 4096, f"first {rows} of 512 activation rows, Q4 and Q8-row, full N and K"
        return make, 512
    if workload == "moe_panels":
        m = synth.c4()
        guq = oracle.pack_q4(m["gu_codes"])
        dq = oracle.pack_q4(m["d_codes"])

        def make(rows):
            X = oracle.x_to_f64(m["x"][:rows], "bf16")
            fn = lambda: oracle.moe(X, m["idx"][:rows], m["w"][:rows], guq, m["gu_scales"], dq, m["d_scales"], 128, 768)
            return fn, rows * 8 * 6.0 * 2048 * 768, f"first {rows} of 32 tokens, full expert chain"
        return make, 32
    if workload == "smallest_q4":
        c = synth.c1()
        wq = oracle.pack_q4(c["codes"])

        def make(rows):
            X = oracle.x_to_f64(c["x"][:rows], "f16")
            return (lambda: oracle.gemm_q4(wq, c["scales"], 256, 512, X)), 2.0 * rows * 256 * 512, \
                f"first {rows} of 16 activation rows"
        return make, 16
    if workload == "denoiser_block":
        gu, dn = synth.c3()
        wgu, wdn = oracle.pack_q4(gu["codes"]), oracle.pack_q4(dn["codes"])

        def make(rows):
            Xg = oracle.x_to_f64(gu["x"][:rows], "bf16")
            Xd = oracle.x_to_f64(dn["x"][:rows], "bf16")

            def fn():
                oracle.gemm_q4(wgu, gu["scales"], gu["N"], gu["K"], Xg)
                oracle.gemm_q4(wdn, dn["scales"], dn["N"], dn["K"], Xd)
            return fn, 2.0 * rows * (gu["N"] * gu["K"] + dn["N"] * dn["K"]), \
                f"first {rows} of 1024 activation rows of both GEMMs (gate/up and down), full N and K"
        return make, 1024
    else:
        T = int(workload.split("_T")[1])
        fmt = "q4" if "q4" in workload else "q8"
        c = synth.c5_q4(T) if fmt == "q4" else synth.c5_q8(T)
    wq = oracle.pack_q4(c["codes"]) if fmt == "q4" else None

    def make(rows):
        X = oracle.x_to_f64(c["x"][:rows], "bf16")
        if fmt == "q4":
            fn = lambda: oracle.gemm_q4(wq, c["scales"], c["N"], c["K"], X)
        else:
            fn = lambda: oracle.gemm_q8row(c["q"], c["rs"], X)
        return fn, 2.0 * rows * c["N"] * c["K"], f"first {rows} of {c['T']} activation rows, full N and K"
    return make, c["T"]


def _calibrated(workload, target_s):
    make, max_rows = _oracle_sample(workload)
    fn, flops, _ = make(1)
    t0 = time.perf_counter()
    fn()
    t1 = max(time.perf_counter() - t0, 1e-4)
    rows = int(max(1, min(max_rows, target_s / t1)))
    return make(rows)


def cpu_baseline(workload):
    fn, flops, desc = _calibrated(workload, 10.0)
    t0 = time.perf_counter()
    fn()
    dt = time.perf_counter() - t0
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle",
            "sample": desc, "seconds": round(dt, 3)}


def run_reference(args, rank, world):
    if rank != 0:
        return
    # each step is a bounded sample, sized so that the whole run takes about two minutes
    per_step = min(20.0, 120.0 / max(1, args.steps + args.warmup))
    fn, flops, desc = _calibrated(args.workload, per_step)
    for _ in range(args.warmup):
        fn()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t0)
    dt = float(np.mean(times))
    v = flops / dt / 1e12
    line = {"impl": "reference", "metric": "dequant-GEMM TFLOP/s (weight GB/s and roofline fraction alongside)",
            "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded)", "config": {"workload": args.workload},
            "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": _cores(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="denoiser_block")
    ap.add_argument("--no-per-config", action="store_true", help="time only the headline workload")
    ap.add_argument("--traffic-pass", action="store_true",
                    help="run every call of the configurations in --configs once (after a warm-up call) and exit")
    ap.add_argument("--configs", default="all", help="comma-separated workloads for --traffic-pass")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time direct calls instead of a captured CUDA graph")
    ap.add_argument("--stream-kernel", type=int, default=0, choices=[0, 1, 2],
                    help="weight-streaming kernel for T <= 16 (CQ_OPT_STREAM_KERNEL): 0 the library's default, "
                         "1 K-split, 2 row-partitioned")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
