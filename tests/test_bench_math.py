"""The benchmark's roofline arithmetic against its definitions (no GPU): layer FLOPs
T * (top_k * 3 * 2 * d * I + 2 * d * E); bytes of the touched experts' weights once (BF16:
2 bytes per weight; FP8: 1 byte per weight plus one FP32 scale per weight row; NVFP4: half a
byte per weight, a scale byte per 16 and an FP32 scale per matrix), the router,
bias, tokens in and out, and the routing outputs; the expert kernel's bytes add its
activation traffic."""
import bench
from sparse_moe_transformer_bias_b300 import workloads as W


def test_layer_flops_and_bytes_bf16():
    s = W.BEAM
    T, n, rows = 16, 89, 128
    flops, bytes_, kern = bench.algorithmic(s, T, n, rows)
    assert flops == T * (8 * 3 * 2 * 5120 * 2560 + 2 * 5120 * 256)
    assert abs(flops / T - 631.77e6) < 0.01e6                     # per-token figure of the layer
    per_expert = 3 * 5120 * 2560 * 2
    assert per_expert == 78_643_200
    assert bytes_ == n * per_expert + 256 * 5120 * 4 + 256 * 4 + 2 * T * 5120 * 2 + T * 8 * 8
    mlp = kern["expert_mlp"]
    assert mlp["flops"] == 2 * rows * 5120 * 2560 * 3
    assert mlp["bytes"] == n * per_expert + rows * (5120 * 2 + 2 * 2560 * 2 + 5120 * 2)


def test_fp8_bytes_count_codes_and_row_scales():
    s = W.BEAM
    _, bytes8, kern8 = bench.algorithmic(s, 16, 89, 128, fp8=True)
    _, bytes16, _ = bench.algorithmic(s, 16, 89, 128)
    per_expert8 = 3 * 5120 * 2560 + (2 * 2560 + 5120) * 4
    assert bytes16 - bytes8 == 89 * (3 * 5120 * 2560 * 2 - per_expert8)
    assert kern8["expert_mlp"]["bytes"] == 89 * per_expert8 + 128 * (5120 * 2 + 2 * 2560 * 2 + 5120 * 2)


def test_nvfp4_bytes_count_codes_scales_and_activation_pieces():
    """NVFP4: half a byte per weight, one E4M3 scale byte per 16 weights and one FP32 tensor
    scale per matrix; x and h move as four NVFP4 pieces (2 bytes of codes and 1/4 byte of
    scales per element), y as BF16."""
    s = W.BEAM
    _, bytes4, kern4 = bench.algorithmic(s, 16, 89, 128, fp4=True)
    _, bytes16, _ = bench.algorithmic(s, 16, 89, 128)
    per_expert4 = 3 * 5120 * 2560 // 2 + 3 * 5120 * 2560 // 16 + 3 * 4
    assert per_expert4 == 22_118_412
    assert bytes16 - bytes4 == 89 * (3 * 5120 * 2560 * 2 - per_expert4)
    act = 128 * (5120 * 2.25 + 2 * 2560 * 2.25 + 5120 * 2)
    assert kern4["expert_mlp"]["bytes"] == 89 * per_expert4 + int(act)


def test_tensor_peaks_follow_the_operand_type():
    assert bench.PEAK_RATIO == {"bf16": 1.0, "fp8": 2.0, "nvfp4": 6.0}   # 2.25 / 4.5 / 13.5 PFLOP/s


def test_single_process_helpers():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.rank_world() == (0, 1, 0)
    name, shape, T, hot = bench.workload("prefill")
    assert (name, T, hot, shape.E) == ("prefill", 4096, 0, 256)
    name, shape, T, _ = bench.workload("decode", n_group=1)
    assert (name, shape.E, shape.topk_group, T) == ("decode_E32", 32, 1, 16)


def test_near_tie_count_flags_only_near_ties():
    """The bench's near-tie diagnostic: a token whose 8th and 9th biased scores differ by
    less than 1e-6, or whose 4th and 5th group scores do, is counted; a token with clear
    gaps is not."""
    import numpy as np
    s = W.BEAM
    bias = np.zeros(s.E, np.float32)
    clear = np.full(s.E, -6.0, np.float32)
    clear[:8] = np.linspace(3.0, 1.0, 8)                 # eight clear picks in group 0
    clear[32::32] = np.linspace(0.5, -1.0, 7)            # one clear leader in each other group
    assert bench.near_tie_count(s, clear[None, :], bias) == 0
    expert_tie = clear.copy()
    expert_tie[8] = expert_tie[7]                         # 9th candidate equal to the 8th pick
    assert bench.near_tie_count(s, expert_tie[None, :], bias) == 1
    group_tie = clear.copy()
    group_tie[4 * 32] = group_tie[3 * 32]                 # 5th group equal to the 4th kept one
    assert bench.near_tie_count(s, np.stack([clear, group_tie, expert_tie]), bias) == 2
