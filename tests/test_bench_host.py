"""Host-side arithmetic of the benchmark (CPU only): the algorithmic bytes
and flops the roofline divides by, checked against counts worked out by
hand for the benchmark's workloads."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench        # noqa: E402
import li_inputs    # noqa: E402


def test_decode_32k_scan_bytes_and_flops():
    w = li_inputs.spec("fp8_32k_b32")
    # 32 x 32768 tokens x (192 fp8 codes + 4-byte scale), fp8 absorbed queries, fp32 weights
    assert bench.scan_bytes(w) == 32 * 32768 * 196 + 32 * 4 * 64 * 192 + 32 * 4 * 64 * 4 == 207_126_528
    assert bench.scan_flops(w) == 2 * 32 * 32768 * 4 * 64 * 192 == 103_079_215_104
    sb = bench.step_bytes(w)
    assert sb["latent"] + sb["lat_scale"] == 205_520_896
    assert sb["total"] == 208_896_000


def test_prefill_flops_count_causal_pairs_only():
    w = li_inputs.spec("prefill_bf16_128k")
    q_pos = list(range(126976, 131072))
    pairs = sum(t + 1 for t in q_pos)
    assert pairs == 528_484_352
    assert bench.scan_flops(w, q_pos) == 2 * pairs * 4 * 64 * 192      # 51.95 TFLOP
    # bf16 latent, no scales, bf16 absorbed queries for 4,096 queries
    assert bench.scan_bytes(w) == 131072 * 192 * 2 + 4096 * 4 * 64 * 192 * 2 + 4096 * 4 * 64 * 4


def test_batch1_8k_flops():
    w = li_inputs.spec("dsa_bf16_8k")
    assert bench.scan_flops(w) == 2 * 8192 * 4 * 64 * 192             # 805 MFLOP


def test_whole_job_rate_units():
    # 208,896,000 bytes in 89 us on one GPU = 2,347 GB/s
    assert abs(bench.whole_job_rate(208_896_000, 1, 0.089) - 2347.146) < 0.01
