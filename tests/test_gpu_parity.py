"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, on a GB300.

Route ids and the align layout are compared bit for bit; route weights within 2e-6;
the layer output element by element within max |y - ref| / max(|ref|, rms(ref)) <= 2e-2.
"""
import numpy as np
import pytest

from expert_gemm_gb300 import workloads as W
from gpu_harness import (TOL, Guarded, align_to_numpy, assert_align_equal, dev_weights, dims_of, inputs, parity_error,
                         to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


@pytest.fixture(scope="module")
def ml(torch):
    from expert_gemm_gb300 import build, moe_lora
    build.build()
    moe_lora.load()
    return moe_lora


def run_case(ml, torch, oracle, wl, block_m=None, tokens=None, logits=None, lora=None, check_route=True):
    logits0, lora0, x, w = inputs(wl)
    logits = logits0 if logits is None else logits
    lora = lora0 if lora is None else lora
    bm = block_m or ml.pick_block_m(wl.T, wl.k, wl.E, wl.L, wl.H, wl.I)
    d = dims_of(wl, bm, ml)
    guards = Guarded(torch)
    layer = guards.guard_layer(ml.Layer(d, dev_weights(w, torch)))
    out = layer.step(to_dev(logits, torch), to_dev(lora, torch), to_dev(x, torch))
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    guards.check()
    ids_o, w_o = oracle.route(logits, wl.k)
    if check_route:
        assert np.array_equal(layer.topk_ids.cpu().numpy(), ids_o)
        assert np.allclose(layer.topk_w.cpu().numpy(), w_o, rtol=0, atol=2e-6)
    al_o = oracle.align(ids_o, lora, wl.E, wl.L, bm)
    assert_align_equal(align_to_numpy(layer.bufs), al_o)
    ref = oracle.forward(x, ids_o, w_o.astype(np.float32), lora, w, tokens)
    y = out.float().cpu().numpy()
    if tokens is not None:
        y = y[tokens]
    elem, norm = parity_error(y, ref)
    assert elem <= TOL, (wl.name, bm, elem, norm)
    return elem, norm, layer


# ----------------------------------------------------------------- configs --

@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "sweep_T1", "sweep_T16", "sweep_T256", "sweep_T4096",
                                  "wide"])
def test_config_full(ml, torch, oracle, name):
    """Every output element of every configuration, at full size, against the fp64
    oracle over all T tokens (prefill: 25,600 tokens, about half a minute on the host
    cores), in the launch configuration the benchmark times (the tile table's block);
    route ids and the align layout bit for bit."""
    oracle.set_threads(0)
    run_case(ml, torch, oracle, W.get(name))


@pytest.mark.parametrize("block_m", [16, 32, 64, 128, 256])
def test_every_block_size(ml, torch, oracle, block_m):
    """Both tile orientations on one layer with several tiles and a ragged tail."""
    wl = W.custom(name="mid", T=200, H=384, I=448, E=6, k=2, L=3, ranks=(16, 32, 8), lora_mode="uniform_with_none")
    run_case(ml, torch, oracle, wl, block_m=block_m)


@pytest.mark.parametrize("block_m", [16, 32])
def test_down_split_k(ml, torch, oracle, block_m):
    """Few tokens over a long I: the weight-streaming down GEMM runs with K split 4 ways,
    each split storing fp32 partial rows that the combine adds in split order."""
    wl = W.custom(name="splitk", T=8, H=256, I=2048, E=4, k=2, L=2, ranks=(16, 32), lora_mode="uniform_with_none")
    run_case(ml, torch, oracle, wl, block_m=block_m)


def test_shrink_split_k(ml, torch, oracle):
    """A long reduction (I = 8192) over few adapter runs: the down shrink splits K (here on
    CUDA cores, 32 slices of 256; the tensor-core split runs in the dense_decode layer);
    the CTA that completes a run adds its fp32 partials in slice order."""
    wl = W.custom(name="shsplit", T=6, H=256, I=8192, E=2, k=1, L=3, ranks=(16, 64, 32), lora_mode="uniform")
    d = dims_of(wl, 16, ml)
    assert ml.plan(d)["shrink_on_cores"] and ml.plan(d)["ksplit"]["shrink_dn"] == 32
    run_case(ml, torch, oracle, wl, block_m=16)


def test_gate_up_split_k(ml, torch, oracle):
    """Few feature tiles: the weight-streaming gate_up splits K, its fp32 partials are
    added in split order before SiLU."""
    wl = W.custom(name="gusplit", T=8, H=1024, I=512, E=2, k=1, L=2, ranks=(16, 32), lora_mode="uniform_with_none")
    run_case(ml, torch, oracle, wl, block_m=16)


@pytest.mark.parametrize("block_m", [16, 128])
def test_dense_multi_lora(ml, torch, oracle, block_m):
    """E=1, k=1: multi-LoRA on one dense SwiGLU MLP (every token, weight 1)."""
    wl = W.custom(name="dense", T=40, H=1024, I=2048, E=1, k=1, L=4, ranks=(16, 32, 16, 32), lora_mode="uniform")
    run_case(ml, torch, oracle, wl, block_m=block_m)


def test_dense_decode_config(ml, torch, oracle):
    """The dense 32B-class MLP at decode size (H=5120, I=25600), every output element; its
    shrinks are tcgen05 tiles split over K (fp32 partials summed by the last split)."""
    wl = W.get("dense_decode")
    p = ml.plan(dims_of(wl, ml.pick_block_m(wl.T, wl.k, wl.E, wl.L, wl.H, wl.I), ml))
    assert not p["shrink_on_cores"] and p["ksplit"]["shrink_gu"] > 1 and p["ksplit"]["shrink_dn"] > 1
    run_case(ml, torch, oracle, wl)


# -------------------------------------------------------------- edge cases --

def test_no_adapter_anywhere(ml, torch, oracle):
    wl = W.get("tiny")
    run_case(ml, torch, oracle, wl, lora=np.full(wl.T, -1, np.int32))


def test_zero_adapters_L0(ml, torch, oracle):
    wl = W.custom(name="l0", T=48, H=256, I=256, E=4, k=2, L=0, ranks=(), lora_mode="none")
    for bm in (16, 128, 256):
        run_case(ml, torch, oracle, wl, block_m=bm)


def test_token_order_gather(ml, torch, oracle):
    """x larger than half the L2 (82 MB): the gather copies in token order in a second
    launch.  Ragged T, several blocks per expert, adapters and no-adapter tokens;
    every output element and the align against the oracle."""
    wl = W.custom(name="bigx", T=20011, H=2048, I=256, E=8, k=2, L=3, ranks=(16, 32, 8),
                  lora_mode="uniform_with_none")
    assert ml.plan(dims_of(wl, 0, ml))["launches_forward"] == 7   # gather + token-order copy + ...
    for bm in (128, 256):
        run_case(ml, torch, oracle, wl, block_m=bm)


def test_cta_pair_invalid_ids(ml, torch, oracle):
    """256-row blocks (CTA pairs) with dropped pairs: stale pair records are rejected."""
    wl = W.custom(name="bad256", T=700, H=256, I=384, E=3, k=2, L=3, ranks=(16, 16, 32), lora_mode="uniform_with_none")
    logits, lora, x, w = inputs(wl)
    ids, tw = oracle.route(logits, wl.k)
    ids[3, 0] = -1
    ids[600, 1] = wl.E
    lora = lora.copy()
    lora[7] = wl.L
    d = dims_of(wl, 256, ml)
    layer = ml.Layer(d, dev_weights(w, torch))
    ml.align(d, to_dev(ids, torch), to_dev(lora, torch), layer.bufs, layer.ws_align)
    ml.forward(d, to_dev(x, torch), to_dev(tw.astype(np.float32), torch), layer.bufs, layer.w, layer.out,
               layer.ws_fwd, layer.status)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    assert_align_equal(align_to_numpy(layer.bufs), oracle.align(ids, lora, wl.E, wl.L, 256))
    ref = oracle.forward(x, ids, tw.astype(np.float32), lora, w)
    elem, norm = parity_error(layer.out.float().cpu().numpy(), ref)
    assert elem <= TOL, (wl.name, elem, norm)


def test_all_tokens_one_expert(ml, torch, oracle):
    """One expert gets every token (many blocks of one expert, several adapters per block)."""
    wl = W.custom(name="hot", T=300, H=256, I=320, E=8, k=1, L=4, ranks=(8, 16, 32, 64), lora_mode="uniform_with_none")
    logits, _, _, _ = inputs(wl)
    logits = logits.copy()
    logits[:, 5] += 100.0
    for bm in (16, 128, 256):
        run_case(ml, torch, oracle, wl, block_m=bm, logits=logits)


@pytest.mark.parametrize("block_m", [16, 64, 128, 256])
def test_ranks_off_the_chunk_grid(ml, torch, oracle, block_m):
    """Ranks 40, 24, 48, 8 in a rank-48 bank: A boxes of 48 and 32 rows, rank chunks
    whose last rows are the bank's zero padding, B rows past r_max read as zero; with
    ragged feature tiles (I = 320, H = 448) in every tile orientation."""
    wl = W.custom(name="rk48", T=160, H=448, I=320, E=4, k=2, L=4, ranks=(40, 24, 48, 8),
                  lora_mode="uniform_with_none")
    assert wl.r_max == 48
    run_case(ml, torch, oracle, wl, block_m=block_m)


# Shapes for both shrink tile forms on 128-row blocks: ranks off the 16-chunk grid, and a
# block with more than 32 adapter runs (the group decode takes them 32 at a time) whose
# rank chunks fill several 16-chunk groups with runs cut at the group boundaries.
SHRINK_FORM_CASES = [
    dict(name="rk48", T=160, H=448, I=320, E=4, k=2, L=4, ranks=(40, 24, 48, 8), lora_mode="uniform_with_none"),
    dict(name="manyruns", T=300, H=320, I=192, E=2, k=1, L=48, ranks=tuple(16 if a % 3 else 48 for a in range(48)),
         lora_mode="uniform_with_none"),
    # ~95 distinct rank-64 adapters per 128-row block: ~380 rank chunks, ~24 groups of a block
    dict(name="allruns", T=600, H=192, I=128, E=2, k=1, L=200, ranks=(64,) * 200, lora_mode="uniform"),
]


@pytest.mark.parametrize("block_m", [128, 256])
@pytest.mark.parametrize("form", [1, 2])
@pytest.mark.parametrize("case", SHRINK_FORM_CASES, ids=lambda c: c["name"])
def test_shrink_tile_forms(ml, torch, oracle, case, form, block_m):
    """The tcgen05 shrink of token-tiled blocks as block-diagonal groups (form 1: rank
    chunks of the runs that reach a 128-row unit, several runs per tile; on 256-row
    blocks a unit is a half, and a run with no rows in the other half writes that half's
    S rows as zeros) and one run per tile (form 2: on 256-row blocks one tile per
    half), against the oracle; align bit for bit.  The shape picks a form by itself; the
    test hook forces each."""
    wl = W.custom(**case)
    ml.debug_set_shrink_tiles(form)
    try:
        assert ml.plan(dims_of(wl, block_m, ml))["shrink_block_diag"] == (form == 1)
        run_case(ml, torch, oracle, wl, block_m=block_m)
    finally:
        ml.debug_set_shrink_tiles(0)


@pytest.mark.parametrize("block_m", [128, 256])
def test_shrink_tile_forms_same_bytes(ml, torch, block_m):
    """Both shrink forms form each S element from the same products summed in the same K
    order in fp32, rounded once: the layer outputs are identical bit for bit."""
    wl = W.custom(**SHRINK_FORM_CASES[1])
    logits, lora, x, w = inputs(wl)
    outs = []
    for form in (1, 2):
        ml.debug_set_shrink_tiles(form)
        try:
            layer = ml.Layer(dims_of(wl, block_m, ml), dev_weights(w, torch))
            outs.append(layer.step(to_dev(logits, torch), to_dev(lora, torch), to_dev(x, torch)).clone())
            torch.cuda.synchronize()
            assert int(layer.status.item()) == 0
        finally:
            ml.debug_set_shrink_tiles(0)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))


def test_shrink_tile_form_hook_rejects_unknown_modes(ml):
    with pytest.raises(ml.MoeLoraError):
        ml.debug_set_shrink_tiles(3)
    assert ml.plan(dims_of(W.get("sweep_T4096"), 128, ml))["shrink_block_diag"]
    assert not ml.plan(dims_of(W.get("wide"), 128, ml))["shrink_block_diag"]
    assert not ml.plan(dims_of(W.get("sweep_T16"), 16, ml))["shrink_block_diag"]   # weight-streaming


@pytest.mark.parametrize("T,k", [(512, 8), (4097, 1)])
def test_align_one_chunk_boundary(ml, torch, oracle, T, k):
    """P = 4096 pairs, the largest batch the one-CTA align takes (layout from the sorted
    keys in shared memory), and P = 4097, the smallest the chunked align takes; many
    experts and Zipf adapters with 10% none, bit-exact against the oracle."""
    wl = W.custom(name=f"edge{T}x{k}", T=T, H=128, I=128, E=64, k=k, L=32, ranks=(16,) * 32,
                  lora_mode="zipf_with_none", bias_std=0.5, none_frac=0.1)
    for bm in (16, 128):
        run_case(ml, torch, oracle, wl, block_m=bm)


@pytest.mark.parametrize("block_m", [16, 32, 64])
def test_shrink_paths_every_weight_streaming_block(ml, torch, oracle, block_m):
    """Both shrinks on every weight-streaming block size.  A handful of runs over a short
    weight stream takes the CUDA-core shrink: runs of several rows, ranks 40 and 8, K
    slices cut ragged (H = 2880 = 11 x 256 + 64, I = 320).  A layer whose gate_up weights
    stream for longer (4 experts of 2 x 4096 x 4096) takes the tcgen05 shrink tiles
    (every output element)."""
    few = W.custom(name="fewruns", T=6, H=2880, I=320, E=3, k=2, L=2, ranks=(40, 8), lora_mode="uniform")
    assert ml.plan(dims_of(few, block_m, ml))["shrink_on_cores"]
    run_case(ml, torch, oracle, few, block_m=block_m)
    big = W.custom(name="bigw", T=200, H=4096, I=4096, E=4, k=1, L=3, ranks=(16, 64, 32), lora_mode="uniform_with_none")
    assert not ml.plan(dims_of(big, block_m, ml))["shrink_on_cores"]
    run_case(ml, torch, oracle, big, block_m=block_m)


def test_single_token(ml, torch, oracle):
    wl = W.custom(name="one", T=1, H=512, I=256, E=16, k=4, L=2, ranks=(16, 16), lora_mode="uniform")
    for bm in (16, 128):
        run_case(ml, torch, oracle, wl, block_m=bm)


def test_invalid_ids_dropped(ml, torch, oracle):
    """Out-of-range expert and adapter ids are dropped and counted, never trapped."""
    wl = W.custom(name="bad", T=40, H=256, I=256, E=8, k=2, L=3, ranks=(16, 16, 16), lora_mode="uniform_with_none")
    logits, lora, x, w = inputs(wl)
    ids, tw = oracle.route(logits, wl.k)
    ids[3, 0] = -1
    ids[5, 1] = wl.E
    lora = lora.copy()
    lora[7] = wl.L
    lora[9] = -5
    d = dims_of(wl, 16, ml)
    layer = ml.Layer(d, dev_weights(w, torch))
    # stale scratch: every int32 of the forward workspace names an in-range row, so a
    # dropped pair's row record points at some real row unless the combine checks it
    rows = int(ml.align_capacity(d)[0])
    ws32 = layer.ws_fwd[: layer.ws_fwd.numel() // 4 * 4].view(torch.int32)
    ws32.copy_(torch.randint(0, rows, ws32.shape, dtype=torch.int32, device="cuda"))
    ids_d, tw_d = to_dev(ids, torch), to_dev(tw.astype(np.float32), torch)
    ml.align(d, ids_d, to_dev(lora, torch), layer.bufs, layer.ws_align)
    ml.forward(d, to_dev(x, torch), tw_d, layer.bufs, layer.w, layer.out, layer.ws_fwd, layer.status)
    torch.cuda.synchronize()
    al = align_to_numpy(layer.bufs)
    assert_align_equal(al, oracle.align(ids, lora, wl.E, wl.L, 16))
    assert al["num_dropped"] == 2 + 2 * 2
    ref = oracle.forward(x, ids, tw.astype(np.float32), lora, w)
    elem, norm = parity_error(layer.out.float().cpu().numpy(), ref)
    assert elem <= TOL, (wl.name, elem, norm)


@pytest.mark.parametrize("case", ["decode_bm16", "gusplit_bm16", "mid_bm128", "mid_bm256", "mid_bm128_bd",
                                  "mid_bm256_bd"])
def test_deterministic_bytes(ml, torch, case):
    """No floating-point atomics on the path: repeated calls give identical output bytes,
    also after another batch has run through the same buffers (K-split partial buffers,
    the bf16 row path, CTA pairs claiming tiles dynamically, and the block-diagonal
    shrink whose group table is counted with integer atomics, all covered)."""
    bd = case.endswith("_bd")
    case = case[:-3] if bd else case
    shapes = {
        "decode": W.get("decode"),
        "gusplit": W.custom(name="gusplit", T=8, H=1024, I=512, E=2, k=1, L=2, ranks=(16, 32),
                            lora_mode="uniform_with_none"),
        "mid": W.custom(name="mid", T=700, H=384, I=448, E=6, k=2, L=3, ranks=(16, 32, 8),
                        lora_mode="uniform_with_none"),
    }
    name, bm = case.split("_bm")
    wl = shapes[name]
    logits, lora, x, w = inputs(wl)
    ml.debug_set_shrink_tiles(1 if bd else 0)
    try:
        layer = ml.Layer(dims_of(wl, int(bm), ml), dev_weights(w, torch))
        lg, lr, xd = to_dev(logits, torch), to_dev(lora, torch), to_dev(x, torch)
        first = layer.step(lg, lr, xd).clone()
        g = np.random.default_rng(9)
        layer.step(to_dev(g.standard_normal(logits.shape).astype(np.float32), torch), lr,
                   to_dev(W.f32_to_bf16_bits(g.standard_normal(x.shape).astype(np.float32)), torch))
        for _ in range(3):
            again = layer.step(lg, lr, xd)
            torch.cuda.synchronize()
            assert torch.equal(first.view(torch.int16), again.view(torch.int16))
    finally:
        ml.debug_set_shrink_tiles(0)
    assert int(layer.status.item()) == 0


@pytest.mark.parametrize("name", ["tiny", "decode", "sweep_T256", "sweep_T4096"])
def test_route_align_matches_separate_calls(ml, torch, name):
    """moe_lora_route_align (one launch up to 4096 pairs, else route + align launches)
    gives the same bytes as moe_lora_route followed by moe_lora_align."""
    wl = W.get(name)
    logits, lora = W.make_routing(wl, 0)
    bm = ml.pick_block_m(wl.T, wl.k, wl.E, wl.L, wl.H, wl.I)
    d = dims_of(wl, bm, ml)
    a_bytes, _ = ml.workspace_size(d)
    lg, lr = to_dev(logits, torch), to_dev(lora, torch)
    res = []
    for fused in (False, True):
        bufs = ml.alloc_align(d)
        ws = torch.empty(max(a_bytes, 256), dtype=torch.uint8, device="cuda")
        ids = torch.full((wl.T, wl.k), -9, dtype=torch.int32, device="cuda")
        tw = torch.full((wl.T, wl.k), -9.0, dtype=torch.float32, device="cuda")
        if fused:
            ml.route_align(d, lg, lr, ids, tw, bufs, ws)
        else:
            ml.route(lg, wl.k, ids, tw)
            ml.align(d, ids, lr, bufs, ws)
        torch.cuda.synchronize()
        res.append((ids.cpu().numpy(), tw.cpu().numpy(), align_to_numpy(bufs)))
    (i0, w0, a0), (i1, w1, a1) = res
    assert np.array_equal(i0, i1)
    assert np.array_equal(w0.view(np.int32), w1.view(np.int32))
    assert_align_equal(a1, a0)


@pytest.mark.parametrize("T,k", [(4, 2), (16, 2), (11, 3), (16, 4), (13, 5)])
def test_align_small_batch_sizes(ml, torch, oracle, T, k):
    """P = 8, 32, 33, 64, 65 pairs (32-, 64- and 128-key sort chunks of the one-CTA align):
    bit-exact against the oracle with invalid expert and adapter ids dropped; the fused
    route+align (T <= 32) gives the same bytes as route then align."""
    wl = W.custom(name=f"w{T}x{k}", T=T, H=128, I=128, E=8, k=k, L=3, ranks=(16, 8, 32),
                  lora_mode="uniform_with_none")
    logits, lora, _, _ = inputs(wl)
    for bm in (16, 128):
        d = dims_of(wl, bm, ml)
        a_bytes, _ = ml.workspace_size(d)
        ids, _ = oracle.route(logits, wl.k)
        ids = ids.copy()
        bad_lora = lora.copy()
        ids[0, 0] = -1
        ids[T - 1, k - 1] = wl.E
        bad_lora[T // 2] = wl.L
        bufs = ml.alloc_align(d)
        ws = torch.empty(max(a_bytes, 256), dtype=torch.int8, device="cuda")
        ml.align(d, to_dev(ids, torch), to_dev(bad_lora, torch), bufs, ws)
        torch.cuda.synchronize()
        al = align_to_numpy(bufs)
        assert_align_equal(al, oracle.align(ids, bad_lora, wl.E, wl.L, bm))
        assert al["num_dropped"] >= 2
        # fused route + align against the separate calls
        lg, lr = to_dev(logits, torch), to_dev(lora, torch)
        res = []
        for fused in (False, True):
            b2 = ml.alloc_align(d)
            w2 = torch.empty(max(a_bytes, 256), dtype=torch.uint8, device="cuda")
            i2 = torch.full((wl.T, wl.k), -9, dtype=torch.int32, device="cuda")
            t2 = torch.full((wl.T, wl.k), -9.0, dtype=torch.float32, device="cuda")
            if fused:
                ml.route_align(d, lg, lr, i2, t2, b2, w2)
            else:
                ml.route(lg, wl.k, i2, t2)
                ml.align(d, i2, lr, b2, w2)
            torch.cuda.synchronize()
            res.append((i2.cpu().numpy(), align_to_numpy(b2)))
        assert np.array_equal(res[0][0], res[1][0])
        assert_align_equal(res[1][1], res[0][1])
        assert_align_equal(res[0][1], oracle.align(oracle.route(logits, wl.k)[0], lora, wl.E, wl.L, bm))


@pytest.mark.parametrize("E", [200, 1000])
def test_route_many_experts(ml, torch, oracle, E):
    """The router's wider register paths (E > 128: 8 and 32 logits per lane): ids bit-exact
    and weights within 2e-6 of the oracle through the fused one-CTA route+align (T = 20)
    and the route kernel (T = 300, and the separate calls), the align from them
    bit-exact."""
    for T in (20, 300):
        wl = W.custom(name=f"re{E}x{T}", T=T, H=64, I=64, E=E, k=8, L=2, ranks=(16, 16),
                      lora_mode="uniform_with_none")
        logits, lora = W.make_routing(wl, 0)
        d = dims_of(wl, 16, ml)
        a_bytes, _ = ml.workspace_size(d)
        ids_o, w_o = oracle.route(logits, wl.k)
        lg, lr = to_dev(logits, torch), to_dev(lora, torch)
        for fused in (False, True):
            bufs = ml.alloc_align(d)
            ws = torch.empty(max(a_bytes, 256), dtype=torch.uint8, device="cuda")
            ids = torch.full((T, wl.k), -9, dtype=torch.int32, device="cuda")
            tw = torch.full((T, wl.k), -9.0, dtype=torch.float32, device="cuda")
            if fused:
                ml.route_align(d, lg, lr, ids, tw, bufs, ws)
            else:
                ml.route(lg, wl.k, ids, tw)
                ml.align(d, ids, lr, bufs, ws)
            torch.cuda.synchronize()
            assert np.array_equal(ids.cpu().numpy(), ids_o), (E, T, fused)
            assert np.allclose(tw.cpu().numpy(), w_o, rtol=0, atol=2e-6), (E, T, fused)
            assert_align_equal(align_to_numpy(bufs), oracle.align(ids_o, lora, E, wl.L, 16))


@pytest.mark.parametrize("E", [64, 128, 200])
def test_route_ties_and_signed_zero(ml, torch, oracle, E):
    """Logits drawn from a handful of values -- exact ties, +0 and -0, -inf -- so every
    selection round meets equal candidates in many lanes.  The router's warp reductions
    must keep the oracle's choice (larger logit; equal ones to the lower expert index;
    -0 equal to +0) bit for bit, through the fused one-CTA route+align (T = 20) and the
    route kernel (T = 300)."""
    vals = np.array([-np.inf, -1.0, -0.0, 0.0, 0.5, 1.0, 1.0], dtype=np.float32)
    g = np.random.default_rng(11)
    for T in (20, 300):
        wl = W.custom(name=f"tie{E}x{T}", T=T, H=64, I=64, E=E, k=8, L=2, ranks=(16, 16), lora_mode="uniform")
        logits = vals[g.integers(0, len(vals), size=(T, E))]
        _, lora = W.make_routing(wl, 0)
        d = dims_of(wl, 16, ml)
        a_bytes, _ = ml.workspace_size(d)
        ids_o, w_o = oracle.route(logits, wl.k)
        lg, lr = to_dev(logits, torch), to_dev(lora, torch)
        for fused in (False, True):
            bufs = ml.alloc_align(d)
            ws = torch.empty(max(a_bytes, 256), dtype=torch.uint8, device="cuda")
            ids = torch.full((T, wl.k), -9, dtype=torch.int32, device="cuda")
            tw = torch.full((T, wl.k), -9.0, dtype=torch.float32, device="cuda")
            if fused:
                ml.route_align(d, lg, lr, ids, tw, bufs, ws)
            else:
                ml.route(lg, wl.k, ids, tw)
            torch.cuda.synchronize()
            assert np.array_equal(ids.cpu().numpy(), ids_o), (E, T, fused)
            assert np.allclose(tw.cpu().numpy(), w_o, rtol=0, atol=2e-6), (E, T, fused)


def test_empty_batch(ml, torch):
    wl = W.get("tiny")
    _, _, _, w = inputs(wl)
    d = dims_of(wl, 16, ml, T=0)
    layer = ml.Layer(d, dev_weights(w, torch))
    e = torch.empty((0, wl.E), dtype=torch.float32, device="cuda")
    layer.step(e, torch.empty(0, dtype=torch.int32, device="cuda"),
               torch.empty((0, wl.H), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert layer.bufs["totals"].cpu().tolist() == [0, 0, 0, 0]
    # the host-buffer entry point with no tokens: nothing in, nothing out, status clean
    assert layer.step_host(torch.empty((0, wl.E), dtype=torch.float32),
                           torch.empty(0, dtype=torch.int32), torch.empty((0, wl.H), dtype=torch.int16),
                           torch.empty((0, wl.H), dtype=torch.int16)) == 0


def test_repeat_calls_reuse_buffers(ml, torch, oracle):
    """Two different batches through one Layer: no state leaks between calls."""
    wl = W.get("tiny")
    e1, _, layer = run_case(ml, torch, oracle, wl)
    logits, lora, x, w = inputs(wl, seed=0)
    g = np.random.default_rng(5)
    logits2 = g.standard_normal(logits.shape).astype(np.float32)
    lora2 = g.integers(-1, wl.L, size=wl.T).astype(np.int32)
    out = layer.step(to_dev(logits2, torch), to_dev(lora2, torch), to_dev(x, torch))
    torch.cuda.synchronize()
    ids, tw = oracle.route(logits2, wl.k)
    ref = oracle.forward(x, ids, tw.astype(np.float32), lora2, w)
    elem, norm = parity_error(out.float().cpu().numpy(), ref)
    assert elem <= TOL, (wl.name, elem, norm)


# ------------------------------------------------------------ host buffers --

@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_layer_host_entry(ml, torch, oracle, name):
    """moe_lora_layer_host: host inputs in, host output back, same result."""
    wl = W.get(name)
    logits, lora, x, w = inputs(wl)
    bm = ml.pick_block_m(wl.T, wl.k, wl.E, wl.L, wl.H, wl.I)
    layer = ml.Layer(dims_of(wl, bm, ml), dev_weights(w, torch))
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()   # noqa: E731
    lg, lr, xh = pin(logits), pin(lora), pin(x.view(np.int16))
    out_h = torch.empty((wl.T, wl.H), dtype=torch.int16).pin_memory()
    dropped = layer.step_host(lg, lr, xh, out_h)
    assert dropped == 0
    y = out_h.view(torch.bfloat16).float().numpy()
    ids, tw = oracle.route(logits, wl.k)
    ref = oracle.forward(x, ids, tw.astype(np.float32), lora, w)
    elem, norm = parity_error(y, ref)
    assert elem <= TOL, (wl.name, elem, norm)


@pytest.mark.parametrize("name", ["decode", "sweep_T4096"])
def test_layer_host_in_place_and_copied_buffers_agree(ml, torch, name):
    """moe_lora_layer_host reads pinned host inputs and writes a pinned host output in
    place (at most 4 MB each) and copies pageable ones: decode's pinned buffers are all
    in place, its pageable ones all copied; at T = 4096 the 16 MB x and out are copied
    while the 2 MB logits are read in place; pinned views 4 bytes off a 16-byte boundary
    are copied.  Every path gives the bytes of the device-buffer step."""
    wl = W.get(name)
    logits, lora, x, w = inputs(wl)
    layer = ml.Layer(dims_of(wl, 0, ml), dev_weights(w, torch))
    ref = layer.step(to_dev(logits, torch), to_dev(lora, torch), to_dev(x, torch)).clone()
    torch.cuda.synchronize()
    ref_h = ref.view(torch.int16).cpu()
    for pinned in (True, False):
        host = lambda a: torch.from_numpy(np.ascontiguousarray(a)).clone()   # noqa: E731
        lg, lr, xh = host(logits), host(lora), host(x.view(np.int16))
        out_h = torch.full((wl.T, wl.H), 0x7fc1, dtype=torch.int16)
        if pinned:
            lg, lr, xh, out_h = lg.pin_memory(), lr.pin_memory(), xh.pin_memory(), out_h.pin_memory()
        assert layer.step_host(lg, lr, xh, out_h) == 0
        assert torch.equal(out_h, ref_h), (name, pinned)
    # pinned but not 16-byte aligned (each view starts 4 bytes into its buffer): copied
    lg_b = torch.empty(logits.size + 1, dtype=torch.float32).pin_memory()
    lg_b[1:].copy_(torch.from_numpy(logits.reshape(-1)))
    x_b = torch.empty(x.size + 2, dtype=torch.int16).pin_memory()
    x_b[2:].copy_(torch.from_numpy(x.view(np.int16).reshape(-1)))
    out_b = torch.full((wl.T * wl.H + 2,), 0x7fc1, dtype=torch.int16).pin_memory()
    lr_h = torch.from_numpy(np.ascontiguousarray(lora)).clone().pin_memory()
    assert layer.step_host(lg_b[1:], lr_h, x_b[2:], out_b[2:]) == 0
    assert torch.equal(out_b[2:].view(wl.T, wl.H), ref_h), name


@pytest.mark.parametrize("name", ["tiny", "decode", "sweep_T256"])
def test_layer_graph_replay(ml, torch, oracle, name):
    """moe_lora_layer_graph_*: the captured host-to-host layer gives moe_lora_layer_host's
    bytes, and a replay after new inputs are written into the same pinned buffers
    computes the new batch."""
    wl = W.get(name)
    logits, lora, x, w = inputs(wl)
    layer = ml.Layer(dims_of(wl, 0, ml), dev_weights(w, torch))
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()   # noqa: E731
    lg, lr, xh = pin(logits), pin(lora), pin(x.view(np.int16))
    out_direct = torch.empty((wl.T, wl.H), dtype=torch.int16).pin_memory()
    layer.step_host(lg, lr, xh, out_direct)
    out_g = torch.empty((wl.T, wl.H), dtype=torch.int16).pin_memory()
    stream = torch.cuda.Stream()
    graph = layer.graph_host(lg, lr, xh, out_g, stream)
    try:
        assert graph.run() == 0
        assert torch.equal(out_g, out_direct)
        g = np.random.default_rng(11)
        logits2 = g.standard_normal(logits.shape).astype(np.float32)
        x2 = W.f32_to_bf16_bits(g.standard_normal(x.shape).astype(np.float32))
        lg.copy_(torch.from_numpy(logits2))
        xh.copy_(torch.from_numpy(x2.view(np.int16)))
        assert graph.run() == 0
        ids, tw = oracle.route(logits2, wl.k)
        ref = oracle.forward(x2, ids, tw.astype(np.float32), lora, w)
        elem, norm = parity_error(out_g.view(torch.bfloat16).float().numpy(), ref)
        assert elem <= TOL, (wl.name, elem, norm)
    finally:
        graph.close()


@pytest.mark.parametrize("block_m", [16, 64, 128, 256])
def test_rank_padding_may_hold_any_finite_values(ml, torch, oracle, block_m):
    """A and B rows at or beyond each adapter's rank are outside the layer.  The kernels
    read them in 16-rank chunks, but the shrinks write S = 0 at those ranks (a select,
    not a product), so finite junk there changes nothing: the device banks get N(0,1)
    junk in every padding row, the oracle sees the clean banks."""
    wl = W.custom(name="pad", T=120, H=320, I=448, E=4, k=2, L=4, ranks=(40, 8, 24, 48),
                  lora_mode="uniform_with_none")
    logits, lora, x, w = inputs(wl)
    dev = {n: to_dev(w[n], torch) for n in ("W_gu", "W_dn", "A_gu", "B_gu", "A_dn", "B_dn")}
    g = torch.Generator(device="cuda").manual_seed(5)
    for name in ("A_gu", "B_gu", "A_dn", "B_dn"):
        t = dev[name]
        for a, r in enumerate(wl.ranks):
            pad = t[a, :, r:, :]
            pad.copy_(torch.randn(pad.shape, generator=g, device="cuda").to(torch.bfloat16))
    d = dims_of(wl, block_m, ml)
    ids, tw = oracle.route(logits, wl.k)
    ref = oracle.forward(x, ids, tw.astype(np.float32), lora, w)
    for form in ((1, 2) if block_m == 128 else (0,)):   # both shrink tile forms of 128-row blocks
        ml.debug_set_shrink_tiles(form)
        try:
            layer = ml.Layer(d, dev)
            out = layer.step(to_dev(logits, torch), to_dev(lora, torch), to_dev(x, torch))
            torch.cuda.synchronize()
        finally:
            ml.debug_set_shrink_tiles(0)
        assert int(layer.status.item()) == 0
        elem, norm = parity_error(out.float().cpu().numpy(), ref)
        assert elem <= TOL, (block_m, form, elem, norm)


def test_align_scan_in_global_memory(ml, torch, oracle):
    """More than 16,384 (expert, adapter) buckets (1024 experts x 17): the chunked align's
    scan keeps its per-bucket arrays in global scratch instead of shared memory; bit-exact
    against the oracle, as the shared-memory scan is in every other chunked case."""
    wl = W.custom(name="nb17k", T=6000, H=64, I=64, E=1024, k=1, L=16, ranks=(16,) * 16,
                  lora_mode="zipf_with_none", bias_std=0.5, none_frac=0.1)
    assert wl.E * (wl.L + 1) > 16384 and wl.T * wl.k > 4096
    logits, lora = W.make_routing(wl, 0)
    ids, _ = oracle.route(logits, wl.k)
    for bm in (16, 128):
        d = dims_of(wl, bm, ml)
        a_bytes, _ = ml.workspace_size(d)
        bufs = ml.alloc_align(d)
        ws = torch.empty(a_bytes, dtype=torch.uint8, device="cuda")
        ml.align(d, to_dev(ids, torch), to_dev(lora, torch), bufs, ws)
        torch.cuda.synchronize()
        assert_align_equal(align_to_numpy(bufs), oracle.align(ids, lora, wl.E, wl.L, bm))
