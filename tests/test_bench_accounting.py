"""The algorithmic work behind the benchmark's roofline figures, on the CPU.

  * Dequant bytes per token: codes d*b/8, one E4M3 byte per group, one pi byte per stage
    and a 16-bit output row, plus every centroid table read once.  For the 1.3B layer
    (INT2, B = 32, T = 2, C = 256) that is 294 B per token plus 8 B of tables amortised over
    32760 tokens, 302 B/token in all.
  * Useful assignment flops: 2 N C d per tensor.
  * Attention over the compressed cache: per key, the key's and the value's codes, scales
    and pi bytes (2 x 38 B at INT2, B = 32, T = 2), each tensor's tables once, the queries
    read and the outputs written.
  * Launches per step: one seeded start, per stage four setup kernels and seven per Lloyd
    round, the encode and the fused dequant: 151 for the 1.3B layer, the count of the ncu
    launch list of one bench step.
"""
import bench
from video_kv_cache_gb300 import synth


def test_dequant_bytes_of_the_1p3b_layer():
    w = synth.workload("layer_1p3b_32760")
    H, N = w.H, w.N
    b = bench.dequant_bytes(H, N, w.C, w.T, w.bits, w.group)
    per_token = 128 * 2 // 8 + 128 // 32 + 2 + 128 * 2
    assert per_token == 294
    assert b == H * (N * per_token + 2 * 256 * 128 * 4)
    assert round(b / (H * N)) == 302
    assert b == 237446016


def test_dequant_bytes_scale_with_tables_and_output_width():
    one = bench.dequant_bytes(1, 1000, 64, 1, 4, 16)
    assert bench.dequant_bytes(1, 1000, 64, 1, 4, 16, out_bytes=4) - one == 1000 * 128 * 2
    assert bench.dequant_bytes(1, 1000, 64, 1, 4, 16, n_tables=3) - one == 2 * 64 * 128 * 4
    assert bench.dequant_bytes(1, 1000, 64, 0, 4, 16) == 1000 * (64 + 8 + 256)


def test_assignment_flops():
    assert bench.assign_flops(24, 32760, 256) == 2.0 * 24 * 32760 * 256 * 128
    assert bench.assign_flops(1, 1, 1) == 256.0


def test_launches_per_step():
    w = synth.workload("layer_1p3b_32760")
    assert bench.launches_per_step(w) == 151
    w4 = synth.workload("dit13b_65536")
    assert bench.launches_per_step(w4) == 1 + 4 * (4 + 7 * 8) + 2


def test_attention_bytes_of_the_1p3b_layer():
    w = synth.workload("layer_1p3b_32760")
    heads, N = w.H // 2, w.N
    b = bench.attention_bytes(heads, N, w.C, w.T, w.bits, w.group, 1)
    per_key = 2 * (32 + 4 + 2)
    assert per_key == 76
    assert b == heads * (N * per_key + 2 * 2 * 256 * 128 * 4) + heads * 128 * (2 + 4)
    # more queries only add their own rows
    assert bench.attention_bytes(heads, N, w.C, w.T, w.bits, w.group, 16) - b == \
        heads * 15 * 128 * 6


def test_cpu_baseline_sample_is_whole_frames():
    # whole frames, at most 8192 tokens a tensor: two of the 13B shape's sixteen 64x64
    # frames, five of the 1.3B layer's 30x52 frames, all of the single-head tensor
    assert bench.cpu_sample_frames(synth.workload("dit13b_65536")) == 2
    assert bench.cpu_sample_frames(synth.workload("layer_1p3b_32760")) == 5
    assert bench.cpu_sample_frames(synth.workload("single_head_4x32x32")) == 4
    assert bench.DEFAULT_WORKLOAD == "dit13b_65536"
