"""bench.py's work definitions on CPU: the algorithmic FLOPs of a layer and
the algorithmic bytes of its HBM-bound stages, against the figures the scope
table of this build states for the Mixtral-shaped layer (T=8192, H=4096,
F=14336, E=8, top-2) and the closed forms behind them."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from token_dispatch_grouped_moe_gb300.configs import CONFIGS  # noqa: E402


def test_layer_flops():
    # 2 T H E (gate) + 6 R H F (routed SwiGLU FFN) + 6 T H F_s (shared expert)
    assert CONFIGS["mixtral"].flops() == 2 * 8192 * 4096 * 8 + 6 * 16384 * 4096 * 14336
    assert round(CONFIGS["mixtral"].flops() / 1e12, 3) == 5.773
    assert round(CONFIGS["qwen2"].flops() / 1e12, 3) == 3.610
    assert round(CONFIGS["dsk-32k"].flops() / 1e12, 3) == 3.410
    assert round(CONFIGS["dsk-1k"].flops() / 1e12, 3) == 0.107


def test_stage_bytes_mixtral():
    by = bench.roofline_stage_bytes(CONFIGS["mixtral"])
    T, H, E, k, R = 8192, 4096, 8, 2, 16384
    # route: x read, the gate read, ids and weights written (67.3 MB)
    assert by["route"] == T * H * 2 + H * E * 2 + T * k * 8
    assert round(by["route"] / 1e6, 1) == 67.3
    # the materialised dispatch as the scope table defines it: every routed row
    # read and written (268 MB); and the least any dispatch moves
    assert by["permute"] == 2 * R * H * 2 == 268435456
    assert by["permute_min"] == T * H * 2 + R * H * 2 + R * 16
    # the separate combine: k fp32 slots read, the bf16 output written (335 MB)
    assert by["combine"] == k * T * H * 4 + T * H * 2
    assert round(by["combine"] / 1e6) == 336


def test_stage_bytes_shared_expert_slot():
    # with a shared expert the combine reads one more fp32 slot per token
    c = CONFIGS["qwen2"]
    assert bench.roofline_stage_bytes(c)["combine"] == (c.k + 1) * c.T * c.H * 4 + c.T * c.H * 2
