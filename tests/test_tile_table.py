"""The compiled-in tile table and the launch plan (host logic only, no GPU).

The shape class is the pairs per expert T*k/E; each workload lands in the row the
table states, block_m = 0 resolves to that row everywhere, and the plan's K splits
and launch counts follow the rules written beside the table.
"""
import pytest

from expert_gemm_gb300 import moe_lora as ml
from expert_gemm_gb300 import workloads as W


def dims(wl, block_m):
    return ml.LayerDims(T=wl.T, H=wl.H, I=wl.I, E=wl.E, k=wl.k, L=wl.L, r_max=wl.r_max, block_m=block_m,
                        ranks=tuple(wl.ranks))


@pytest.fixture(scope="module", autouse=True)
def lib():
    from expert_gemm_gb300 import build
    build.build()
    return ml.load()


# (name, block_m the table must pick)
EXPECTED = [("tiny", 16), ("decode", 16), ("prefill", 256), ("wide", 256), ("dense_decode", 16),
            ("sweep_T1", 16), ("sweep_T16", 16), ("sweep_T256", 16), ("sweep_T4096", 128)]


@pytest.mark.parametrize("name,bm", EXPECTED)
def test_class_of_each_workload(name, bm):
    wl = W.get(name)
    assert ml.pick_block_m(wl.T, wl.k, wl.E, wl.L, wl.H, wl.I) == bm
    p = ml.plan(dims(wl, 0))
    assert p["block_m"] == bm
    assert p["weight_streaming"] == (bm < 128)


def test_class_boundaries():
    """Pairs per expert above 24, 95 and 2047 move to the next row (short adapter runs:
    255 adapters, so fewer than 20 pairs per (expert, adapter) bucket below 2048); the
    32-row tile is no class of its own.  Experts of the sweep layer (9.4 MB) are far below
    the L2."""
    E, k, L = 8, 1, 255
    for ppe, bm in [(1, 16), (10, 16), (11, 16), (24, 16), (25, 64), (95, 64), (96, 128), (2047, 128), (2048, 256),
                    (5000, 256)]:
        assert ml.pick_block_m(ppe * E, k, E, L) == bm, (ppe, bm)
        assert ml.pick_block_m(ppe * E, k, E, L, 2048, 768) == bm, (ppe, bm)
    assert ml.pick_block_m(0, 1, 8) == 16


def test_experts_larger_than_the_l2_take_the_smallest_tile_that_holds_their_pairs():
    """A dense MLP of H = 5120, I = 25600 (786 MB of bf16 weights) streams from DRAM once
    per block of it: up to 128 pairs per expert the smallest of 16/32/64/128 rows that
    holds them, the table beyond; without H and I the rule is left out."""
    H, I = 5120, 25600
    for T, bm in [(1, 16), (16, 16), (17, 32), (32, 32), (33, 64), (64, 64), (65, 128), (128, 128), (129, 128),
                  (3000, 256)]:
        assert ml.pick_block_m(T, 1, 1, 8, H, I) == bm, (T, bm)
    assert ml.pick_block_m(32, 1, 1, 8) == 64
    # the wide layer's experts (270 MB): 8 experts, top-2
    assert ml.pick_block_m(100, 2, 8, 32, 4096, 11008) == 32
    assert ml.pick_block_m(4096, 2, 8, 32, 4096, 11008) == 256
    # the decode layer's experts (50 MB) stay on the table
    assert ml.pick_block_m(256, 4, 32, 8, 2880, 2880) == 64


def test_long_runs_take_256_row_blocks_from_768_pairs_per_expert():
    """From 768 pairs per expert, 256-row blocks when the pairs per (expert, adapter-or-none
    bucket) T*k / (E*(L+1)) reach 20: no adapters, or few adapters for many tokens."""
    E, k = 8, 1
    for ppe, L, bm in [(767, 0, 128), (768, 0, 256), (1500, 0, 256), (768, 37, 256), (768, 38, 128),
                       (1024, 32, 256), (1024, 64, 128), (96, 0, 128)]:
        assert ml.pick_block_m(ppe * E, k, E, L) == bm, (ppe, L, bm)


@pytest.mark.parametrize("name", [n for n, _ in EXPECTED])
def test_auto_block_m_resolves_everywhere(name):
    """block_m = 0 gives the same capacities, workspace sizes and plan as the explicit pick."""
    wl = W.get(name)
    bm = ml.pick_block_m(wl.T, wl.k, wl.E, wl.L, wl.H, wl.I)
    a, b = dims(wl, 0), dims(wl, bm)
    assert ml.align_capacity(a) == ml.align_capacity(b)
    assert ml.workspace_size(a) == ml.workspace_size(b)
    assert ml.layer_workspace_size(a) == ml.layer_workspace_size(b)
    assert ml.plan(a) == ml.plan(b)


def test_decode_plan():
    """Decode layer (64 pairs over 32 experts, H = I = 2880): 16-token weight-streaming
    tiles; the down GEMM (12 feature tiles per block) splits K two ways to give each
    of the 152 SMs about three tiles; gate_up (23 tiles per block) needs no split; the
    2880-long shrinks stay whole (45 K-tiles < 64)."""
    p = ml.plan(dims(W.get("decode"), 0))
    assert p["ksplit"] == {"shrink_gu": 1, "gate_up": 1, "shrink_dn": 1, "down": 2}
    assert p["k_tile"] == {"shrink_gu": 64, "gate_up": 64, "shrink_dn": 64, "down": 64}
    assert p["launches_route_align"] == 1
    assert p["launches_forward"] == 6      # gather, 2 shrinks, gate_up, down, combine


def test_route_align_launches():
    """Route and align fuse into one single-CTA launch only for a few tokens (T <= 32 and
    one sort chunk); larger one-chunk batches launch the route kernel, then the one-CTA
    align; more than 4096 pairs take the chunked align (route + chunk/scan/scatter)."""
    assert ml.plan(dims(W.get("decode"), 0))["launches_route_align"] == 1      # T = 16
    assert ml.plan(dims(W.get("sweep_T16"), 0))["launches_route_align"] == 1   # T = 16, 128 pairs
    assert ml.plan(dims(W.get("sweep_T256"), 0))["launches_route_align"] == 2  # 2048 pairs
    assert ml.plan(dims(W.get("tiny"), 0))["launches_route_align"] == 2        # T = 64
    assert ml.plan(dims(W.get("sweep_T4096"), 0))["launches_route_align"] == 4


def test_shrink_on_cores_only_for_a_handful_of_runs_over_a_short_stream():
    """A single token over 128 experts (8 runs, 50 MB of gate_up weights): the shrinks run
    on CUDA cores in 256-wide K slices (H = 2048: 8, I = 768: 3).  Decode, the 64-token
    layer and dense_decode keep tcgen05 shrink tiles (long weight streams or tens of
    runs)."""
    p = ml.plan(dims(W.get("sweep_T1"), 0))
    assert p["shrink_on_cores"] and p["ksplit"]["shrink_gu"] == 8 and p["ksplit"]["shrink_dn"] == 3
    assert p["k_tile"]["shrink_gu"] == 256
    for name in ("decode", "tiny", "dense_decode", "sweep_T16"):
        assert not ml.plan(dims(W.get(name), 0))["shrink_on_cores"], name


def test_prefill_plan():
    p = ml.plan(dims(W.get("prefill"), 0))
    assert p["block_m"] == 256 and not p["weight_streaming"]
    assert p["stages"]["gate_up"] == 6 and p["stages"]["down"] == 6   # 32 KB stages of a CTA pair + 16 KB output staging
    assert p["ksplit"] == {"shrink_gu": 1, "gate_up": 1, "shrink_dn": 1, "down": 1}
    assert p["launches_route_align"] == 4  # 102400 pairs: route, then chunk/scan/scatter
    assert p["launches_forward"] == 7      # the gather copies in token order: a second launch


def test_split_plans():
    """Shapes the GPU tests use to exercise each K split."""
    gu = W.custom(name="gusplit", T=8, H=1024, I=512, E=2, k=1, L=2, ranks=(16, 32), lora_mode="uniform_with_none")
    p = ml.plan(dims(gu, 16))
    assert p["ksplit"]["gate_up"] > 1 and p["ksplit"]["down"] == 1   # I = 512: 8 K-tiles, too few to split
    assert p["launches_forward"] == 7      # + the SiLU pass after the split gate_up
    sh = W.custom(name="shsplit", T=6, H=256, I=8192, E=2, k=1, L=3, ranks=(16, 64, 32), lora_mode="uniform")
    p = ml.plan(dims(sh, 16))
    assert p["ksplit"]["shrink_dn"] > 1 and p["ksplit"]["shrink_gu"] == 1
    l0 = W.custom(name="l0", T=48, H=256, I=256, E=4, k=2, L=0, ranks=(), lora_mode="none")
    p = ml.plan(dims(l0, 16))
    assert p["ksplit"]["shrink_gu"] == 0 and p["ksplit"]["shrink_dn"] == 0
    assert p["launches_forward"] == 4


def test_every_compiled_block_size_has_a_plan():
    wl = W.get("decode")
    for bm in (16, 32, 64, 128, 256):
        p = ml.plan(dims(wl, bm))
        assert p["block_m"] == bm and all(s >= 2 for s in p["stages"].values())
    with pytest.raises(ml.MoeLoraError):
        ml.plan(dims(wl, 48))


def test_deep_ring_for_a_few_pairs():
    """16-token tiles run gate_up and down with a 6-deep ring for batches of at most 32
    pairs (a single token of top-8), and with 3 stages (two CTAs per SM) above."""
    one = ml.plan(dims(W.get("sweep_T1"), 0))
    assert one["block_m"] == 16 and one["stages"]["gate_up"] == 6 and one["stages"]["down"] == 6
    for name in ("decode", "sweep_T16"):
        p = ml.plan(dims(W.get(name), 0))
        assert p["block_m"] == 16 and p["stages"]["gate_up"] == 3 and p["stages"]["down"] == 3
    wl = W.custom(name="four", T=4, H=256, I=256, E=16, k=8, L=2, ranks=(16, 16), lora_mode="uniform")
    assert ml.plan(dims(wl, 16))["stages"]["gate_up"] == 6
    wl = W.custom(name="five", T=5, H=256, I=256, E=16, k=8, L=2, ranks=(16, 16), lora_mode="uniform")
    assert ml.plan(dims(wl, 16))["stages"]["gate_up"] == 3
