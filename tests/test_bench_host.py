"""Host logic of the benchmark, without a GPU: the per-call roofline entry
(bound from the arithmetic intensity, fractions of both measured peaks) and
the DRAM-traffic table read from the committed ncu summary, which is ignored
once the kernel sources differ from those it was taken on."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1600.0, "source": "test"}


def _call(flops, wbytes, other):
    c = bench.Call("c", None, flops, wbytes, other)
    c.launches = 1
    return c


def test_roofline_entry_picks_the_lower_roofline():
    # 2*8*8192*8192 FLOP over 37.7 MB: intensity ~28 flop/B, far below the ridge (300) -> HBM
    c = _call(2.0 * 8 * 8192 * 8192, 8192 * 8192 * 9 // 16, 8 * 8192 * 4)
    e = bench.roofline_entry(c, 0.010, PEAKS, None)
    assert e["bound"] == "hbm" and e["frac"] == e["frac_hbm"]
    assert abs(e["bytes_gbs"] - (c.weight_bytes + c.other_bytes) / 1e-5 / 1e9) < 0.1
    assert abs(e["frac_hbm"] - e["bytes_gbs"] / 6000.0) < 1e-4
    # T=512, K=N=4096: ~960 flop/B -> tensor
    c = _call(2.0 * 512 * 4096 * 4096, 4096 * 4096 * 9 // 16, 512 * 4096 * 6)
    e = bench.roofline_entry(c, 0.020, PEAKS, 123)
    assert e["bound"] == "tensor" and e["frac"] == e["frac_tensor"] and e["traffic"] == 123
    assert abs(e["tflops"] - 2.0 * 512 * 4096 * 4096 / 2e-5 / 1e12) < 0.01


def test_traffic_table_keyed_to_the_kernel_sources(tmp_path):
    h = bench.kernel_sources_hash()
    body = ("| workload | call | launches | DRAM bytes per call | algorithmic bytes |\n"
            "|---|---|---|---|---|\n"
            "| `sweep_q4_T8` | `T8 q4->bf16` | 1 | 37,912,064 | 37,879,808 |\n"
            "| `denoiser_block` | `down q4->bf16` | 2 | 61,000,000 | 60,000,000 |\n")
    p = tmp_path / "t.md"
    p.write_text(f"kernel sources `{h}`\n\n" + body)
    t = bench.load_traffic(str(p))
    assert t[("sweep_q4_T8", "T8 q4->bf16")] == 37912064
    assert t[("denoiser_block", "down q4->bf16")] == 61000000
    p.write_text("kernel sources `0123456789abcdef`\n\n" + body)
    assert bench.load_traffic(str(p)) == {}
    assert bench.load_traffic(str(tmp_path / "missing.md")) == {}


def test_per_config_covers_every_configuration():
    names = set(bench.PER_CONFIG)
    assert {"smallest_q4", "prefill_projection_4096", "moe_panels"} <= names
    for f in ("q4", "q8"):
        for t in (1, 8, 32, 128, 512, 2048):
            assert f"sweep_{f}_T{t}" in names
