"""The launch w4_gemv makes for every workload shape, pinned (GB300, 152 SMs).

The split, the arithmetic and the residency rules of the cluster split
(plan_gemv, gemv_shape in w4_gemv.cu) are thresholds fitted to timings on this
GPU; pinning the plan each workload shape gets means that a change of any
threshold shows up here as a test difference, not as a silent reroute of a
shape to a slower branch.  Fields: (K splits, zero point folded, grid x, grid
y, persistent grid, programmatic dependent launch, shared memory capped,
ring stages, wide x prologue, blocks per SM the instance is built for).
"""
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

FIELDS = ("k_splits", "zero_point_folded", "grid_x", "grid_y", "persistent", "overlap", "capped",
          "ring_stages", "wide_prologue", "blocks_per_sm_max")

PINS = {
    ("single.896x896", 1, 896, 896): (6, 0, 7, 6, 0, 1, 1, 6, 0, 3),
    ("single.896x896", 8, 896, 896): (6, 0, 7, 6, 0, 1, 1, 6, 0, 3),
    ("qwen0.5b.qkv", 1, 896, 1152): (6, 0, 9, 6, 0, 1, 1, 6, 0, 3),
    ("qwen0.5b.qkv", 8, 896, 1152): (6, 0, 9, 6, 0, 1, 1, 6, 0, 3),
    ("qwen0.5b.o", 1, 896, 896): (6, 0, 7, 6, 0, 1, 1, 6, 0, 3),
    ("qwen0.5b.o", 8, 896, 896): (6, 0, 7, 6, 0, 1, 1, 6, 0, 3),
    ("qwen0.5b.gate_up", 1, 896, 9728): (2, 0, 76, 2, 0, 1, 0, 6, 0, 3),
    ("qwen0.5b.gate_up", 8, 896, 9728): (2, 0, 76, 2, 0, 1, 0, 6, 0, 3),
    ("qwen0.5b.down", 1, 4864, 896): (8, 0, 7, 8, 0, 1, 1, 6, 0, 3),
    ("qwen0.5b.down", 8, 4864, 896): (8, 0, 7, 8, 0, 1, 1, 6, 0, 3),
    ("qwen7b.qkv", 1, 3584, 4608): (6, 0, 36, 6, 0, 1, 1, 6, 0, 3),
    ("qwen7b.qkv", 8, 3584, 4608): (6, 0, 36, 6, 0, 1, 1, 6, 0, 3),
    ("qwen7b.o", 1, 3584, 3584): (8, 0, 28, 8, 0, 1, 1, 6, 0, 3),
    ("qwen7b.o", 8, 3584, 3584): (8, 0, 28, 8, 0, 1, 1, 6, 0, 3),
    ("qwen7b.gate_up", 1, 3584, 37888): (1, 1, 296, 1, 0, 1, 1, 6, 0, 3),
    ("qwen7b.gate_up", 8, 3584, 37888): (1, 1, 296, 1, 0, 1, 1, 6, 1, 2),
    ("qwen7b.down", 1, 18944, 3584): (8, 1, 28, 8, 0, 1, 1, 6, 0, 3),
    ("qwen7b.down", 8, 18944, 3584): (8, 1, 28, 8, 0, 1, 1, 6, 1, 2),
    ("27b.up", 1, 5120, 17408): (2, 1, 136, 2, 0, 1, 1, 6, 0, 3),
    ("27b.up", 2, 5120, 17408): (2, 1, 136, 2, 0, 1, 1, 6, 0, 3),
    ("27b.up", 4, 5120, 17408): (2, 1, 136, 2, 0, 1, 1, 5, 0, 3),
    ("27b.up", 5, 5120, 17408): (2, 1, 136, 2, 0, 1, 1, 5, 1, 3),
    ("27b.up", 8, 5120, 17408): (2, 1, 136, 2, 0, 1, 1, 6, 1, 2),
    ("27b.down", 1, 17408, 5120): (6, 1, 40, 6, 0, 1, 1, 6, 0, 3),
    ("27b.down", 2, 17408, 5120): (6, 1, 40, 6, 0, 1, 1, 6, 0, 3),
    ("27b.down", 4, 17408, 5120): (6, 1, 40, 6, 0, 1, 1, 5, 0, 3),
    ("27b.down", 5, 17408, 5120): (6, 1, 40, 6, 0, 1, 1, 6, 1, 2),
    ("27b.down", 8, 17408, 5120): (6, 1, 40, 6, 0, 1, 1, 6, 1, 2),
    ("qwen7b.lm_head", 1, 3584, 152064): (1, 1, 1188, 1, 0, 1, 0, 6, 0, 3),
    ("qwen7b.lm_head", 8, 3584, 152064): (1, 1, 304, 1, 1, 1, 0, 6, 0, 2),
}


@pytest.mark.parametrize("key", sorted(PINS), ids=lambda k: f"{k[0]}-M{k[1]}")
def test_launch_plan_pinned(key):
    from int4_weight_only_w4_gb300 import w4
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("pins are for a 152-SM GB300")
    name, M, K, N = key
    plan = w4.gemv_plan(M, K, N)
    got = tuple(int(plan[f]) for f in FIELDS)
    assert got == PINS[key], dict(zip(FIELDS, got))
    # w4_gemv_config reports the same split and arithmetic, independent of M
    _, S, fold = w4.gemv_config(K, N)
    assert (S, int(fold)) == PINS[key][:2]
