"""The roofline numerator bench.py reports (algorithmic bytes and flops of one
layer forward), pinned to figures worked out independently of its formula.

Per expert the weights are w13 [2I, H] and w2 [H, I] plus, for the group-128
formats, one fp16 scale (and with zero points one byte) per 128 weights along
K; fp8 adds two fp32 per-expert scales.  The layer moves the touched experts'
weights, x in (bf16), out (bf16) and the fp32 logits, and does 6 * k * H * I
flops per token (three GEMMs of 2 * H * I flops per routed slot).
"""
import pytest

import bench
from synth import SHAPES

MB = 1e6

# bytes per expert (weights + scales) and flops per token, rounded as printed in
# the workload table these shapes come from: tiny 0.79 MB / 1.57 M, Mixtral
# 352.3 MB / 704.6 M, Qwen2 27.5 MB / 440.4 M, DeepSeek-V3 22.7 MB / 704.6 M,
# Llama-4-Scout 251.7 MB / 251.7 M
# (value, half a unit of its last printed digit), MB and Mflop
TABLE = {
    "tiny": ((0.79, 0.005), (1.57, 0.005)),
    "mixtral": ((352.3, 0.05), (704.6, 0.05)),
    "qwen2": ((27.5, 0.05), (440.4, 0.05)),
    "dsv3": ((22.7, 0.05), (704.6, 0.05)),
    "scout": ((251.7, 0.05), (251.7, 0.05)),
}


@pytest.mark.parametrize("name", sorted(TABLE))
def test_per_expert_bytes_and_per_token_flops(name):
    shape = SHAPES[name]
    (mb, mb_tol), (mflop, mflop_tol) = TABLE[name]
    # one touched expert, no tokens: the weight bytes of one expert alone
    B1, _ = bench.layer_bytes_flops(shape, 0, 1)
    assert abs(B1 / MB - mb) <= mb_tol
    _, F = bench.layer_bytes_flops(shape, 1, 1)
    assert abs(F / 1e6 - mflop) <= mflop_tol


def test_bytes_count_touched_experts_tokens_and_logits():
    s = SHAPES["mixtral"]
    T = 4096
    B, F = bench.layer_bytes_flops(s, T, 8)
    weights = 8 * 3 * s.H * s.I * 2
    assert B == weights + T * s.H * 2 * 2 + T * s.E * 4
    assert F == 6 * s.top_k * s.H * s.I * T
    # two touched experts at T = 1 (Mixtral decode): 0.705 GB
    B1, _ = bench.layer_bytes_flops(s, 1, 2)
    assert B1 / 1e9 == pytest.approx(0.705, abs=0.001)


def test_quantised_formats_count_their_scales_and_zero_points():
    d, awq, w8 = SHAPES["dsv3"], SHAPES["dsv3_awq"], SHAPES["mixtral_w8"]
    n = 3 * d.H * d.I
    assert bench.layer_bytes_flops(d, 0, 1)[0] == n // 2 + n // 128 * 2
    assert bench.layer_bytes_flops(awq, 0, 1)[0] == n // 2 + n // 128 * 3
    m = 3 * w8.H * w8.I
    assert bench.layer_bytes_flops(w8, 0, 1)[0] == m + m // 128 * 2


def test_job_throughput_counts_every_replica_over_the_slowest_rank():
    assert bench.job_throughput(1, 4096, 2.0) == pytest.approx(2.048e6)
    assert bench.job_throughput(4, 4096, 2.0) == pytest.approx(4 * 2.048e6)


def test_clock_sampler_keeps_raw_samples_only_where_asked(tmp_path, monkeypatch):
    # without a log directory the raw samples live in a temporary file removed by
    # the summary; with one they stay there (no GPU needed: without nvidia-smi the
    # summary says so)
    import os
    monkeypatch.delenv("MOE_CLOCK_LOG_DIR", raising=False)
    c = bench.ClockSampler(0)
    with c:
        pass
    c.summary()
    assert not os.path.exists(c.path)
    monkeypatch.setenv("MOE_CLOCK_LOG_DIR", str(tmp_path))
    c = bench.ClockSampler(1)
    with c:
        pass
    c.summary()
    assert c.path == str(tmp_path / "clocks_rank1.csv")
