"""The bench's roofline arithmetic on the five workloads (host only): which resource bounds each decode,
its ideal time, and the fraction a given kernel time reaches."""
import pytest

import bench
from synthetic import gen

PEAKS = {"hbm_gbs": 6688.5, "bf16_tflops": 1875.0, "bf16_tflops_sustained": 1715.2, "sm_max_mhz": 2070.0}


@pytest.mark.parametrize("name,bound,ideal_us", [
    ("llama2-7b-rope-fp16-b1-t4k", "hbm", 5.33),               # 35.65 MB over 6688.5 GB/s
    ("llama2-7b-rope-bf16-b8-t32k", "hbm", 321.4),             # 2.15 GB
    ("llama2-7b-absorbed-fp16-b4-t64k", "hbm", 321.4),
    ("llama2-7b-rope-int4-hadamard-b4-t64k", "tensor", 295.5),  # 554 GFLOP over 1875 TFLOP/s
])
def test_bound_and_ideal_time(name, bound, ideal_us):
    cfg = bench.config_of(name)
    r = bench.roofline_for(cfg, bench.step_work(cfg), 1.0, PEAKS, "test", long_step=False)
    assert r["bound"] == bound
    assert abs(r["roofline_us"] - ideal_us) / ideal_us < 0.01
    # a kernel at exactly the ideal time reaches 1.0
    r1 = bench.roofline_for(cfg, bench.step_work(cfg), r["roofline_us"] / 1e3, PEAKS, "test", long_step=False)
    assert abs(r1["frac"] - 1.0) < 1e-3


def test_joint_absorbed_decode_is_bound_by_the_cuda_cores():
    # 32 heads over one latent stream: the score and p.H_v arithmetic outweighs the bytes
    cfg = gen.ABSORBED_FP16.with_(group_size=32)
    r = bench.roofline_for(cfg, bench.step_work(cfg), 0.377, PEAKS, "test", long_step=False)
    assert r["bound"] == "alu" and abs(r["peak"] - 80.5) < 0.1
    assert abs(bench.alu_peak_tflops(PEAKS) - 152 * 128 * 2 * 2.07e9 / 1e12) < 1e-9


def test_latent_bytes_per_token():
    assert bench.latent_bytes_per_token(gen.ROPE_FP16) == 8192
    assert bench.latent_bytes_per_token(gen.ROPE_INT4) == 2080
    assert bench.latent_bytes_per_token(gen.ROPE_FP16.with_(v_dtype="int4")) == 8 * 512 + 8 * 130
