"""Host-side accounting of bench.py: the FLOP count the throughput metric
divides by, and how a step's projections are grouped into launches.

The algorithmic work of a projection is 2 * T * out * in (one multiply and
one add per weight and token row); the layer totals below are those of
the workload definitions (Qwen3-1.7B-shaped layer at T = 2048: 206.16
GFLOP; Qwen3-8B-shaped layer at T = 8192: 3161 GFLOP)."""
import pytest

import bench
import synth
from synth import workloads


def layer_of(name, only=None):
    layer = object.__new__(bench.Layer)     # the accounting needs no tensors
    layer.wl = workloads.WORKLOADS[name]
    layer.T = layer.wl["T"]
    layer.only = only
    return layer


def test_layer_flops_match_the_workload_totals():
    assert layer_of("qwen3_1p7b_q4k_t2048").flops() / 1e9 == pytest.approx(206.16, abs=0.01)
    assert layer_of("qwen3_8b_q2k_q6k_t8192").flops() / 1e9 == pytest.approx(3161.1, abs=0.05)


def test_flops_of_a_subset_and_of_one_projection():
    layer = layer_of("qwen3_8b_q2k_q6k_t8192")
    # down: 4096 x 12288 at T = 8192
    assert layer.flops(idx=[6]) == 2 * 8192 * 4096 * 12288
    assert layer_of("qwen3_8b_q2k_q6k_t8192", only="down").flops() == 2 * 8192 * 4096 * 12288
    assert sum(layer.flops(idx=[i]) for i in range(7)) == layer.flops()


def test_grouped_launches_follow_runs_of_one_type():
    layer = layer_of("qwen3_8b_q2k_q6k_t8192")
    assert layer.launches(grouped=True) == [(synth.Q2_K, [0, 1, 2, 3, 4, 5]), (synth.Q6_K, [6])]
    assert layer.launches(grouped=False) == [(synth.Q2_K, [i]) for i in range(6)] + [(synth.Q6_K, [6])]
    assert layer_of("qwen3_1p7b_q4k_t2048").launches() == [(synth.Q4_K, list(range(7)))]


def test_a_launch_takes_at_most_eight_projections():
    layer = object.__new__(bench.Layer)
    layer.wl = {"T": 16, "projections": [("p%d" % i, 256, 256, "h", synth.Q8_0) for i in range(11)]}
    layer.T, layer.only = 16, None
    assert [len(idx) for _, idx in layer.launches()] == [8, 3]


def test_only_filter_keeps_one_projection():
    assert layer_of("qwen3_8b_q2k_q6k_t8192", only="gate").launches() == [(synth.Q2_K, [4])]
