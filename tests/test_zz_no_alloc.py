"""moe_lora_align_static: the align entry point that allocates nothing.

Some callers cannot allocate device memory when they call: serving engines that
give almost all HBM to their own pool, and decode loops that must not pay for a
cudaMalloc (which may synchronise the device).  moe_lora_align_static runs the
same align kernels with their scratch in the library's static device array.
These tests check, through the C ABI, that it returns exactly what moe_lora_align
returns with a caller workspace -- on two calls in a row, since every call reuses
the same array -- and that it refuses sizes beyond the array.

This file is collected last on purpose and needs no fixture from other files.
"""
import numpy as np
import pytest

from expert_gemm_gb300 import workloads as W


@pytest.fixture(scope="module")
def ml():
    from expert_gemm_gb300 import build, moe_lora
    build.build()
    moe_lora.load()
    return moe_lora


def _dims(ml, wl, bm):
    return ml.LayerDims(T=wl.T, H=wl.H, I=wl.I, E=wl.E, k=wl.k, L=wl.L, r_max=wl.r_max, block_m=bm, ranks=wl.ranks)


def test_static_scratch_size_is_enforced(ml):
    """Dims whose align scratch is larger than the static array are refused on the host."""
    big = ml.LayerDims(T=1 << 20, H=64, I=64, E=1024, k=8, L=64, r_max=16, block_m=128, ranks=(16,) * 64)
    need, _ = ml.workspace_size(big)
    assert need > ml.STATIC_SCRATCH_BYTES
    bufs = {n: np.zeros(16, dtype=np.int32) for n in ("sorted_p", "expert_begin", "block_expert", "block_runs",
                                                      "runs", "totals")}
    with pytest.raises(ml.MoeLoraError) as ei:
        ml.align_static(big, np.zeros(16, np.int32), np.zeros(16, np.int32), bufs, stream=0)
    assert ei.value.status == ml.EWORKSPACE


def _route(ml, torch, wl, seed):
    logits, lora = W.make_routing(wl, seed)
    lg = torch.from_numpy(logits).cuda()
    lr = torch.from_numpy(lora).cuda()
    ids = torch.empty((wl.T, wl.k), dtype=torch.int32, device="cuda")
    tw = torch.empty((wl.T, wl.k), dtype=torch.float32, device="cuda")
    ml.route(lg, wl.k, ids, tw)
    return ids, lr


def _compare(ml, torch, wl, d, ids, lr):
    ref = ml.alloc_align(d)
    got = ml.alloc_align(d)
    for t in got.values():
        t.fill_(-7)
    a_bytes, _ = ml.workspace_size(d)
    ws = torch.empty(a_bytes, dtype=torch.uint8, device="cuda")
    ml.align(d, ids, lr, ref, ws)
    ml.align_static(d, ids, lr, got)
    torch.cuda.synchronize()
    tot = ref["totals"].cpu().tolist()
    assert got["totals"].cpu().tolist() == tot
    rows, nb, nr, _ = tot
    for name, n in (("sorted_p", rows), ("block_expert", nb), ("block_runs", nb + 1), ("runs", nr),
                    ("expert_begin", wl.E + 1)):
        assert torch.equal(got[name][:n].cpu(), ref[name][:n].cpu()), (wl.name, name)


@pytest.mark.gpu
def test_align_static_matches_align_twice(ml):
    """Two calls in a row on each layer, a different routing each time: bit-identical to
    moe_lora_align.  decode and sweep_T256 (at most 4096 pairs) take the one-CTA align;
    sweep_T4096 (32,768 pairs over 128 x 65 buckets) and wide (8,192 pairs) take the
    chunked align, whose sort keys, per-chunk bucket counts and bucket bases live in
    the static array, so the second call runs over the first call's leftovers."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    for name in ("decode", "sweep_T256", "sweep_T4096", "wide"):
        wl = W.get(name)
        bm = ml.pick_block_m(wl.T, wl.k, wl.E, wl.L, wl.H, wl.I)
        d = _dims(ml, wl, bm)
        a_bytes, _ = ml.workspace_size(d)
        assert a_bytes <= ml.STATIC_SCRATCH_BYTES
        if name in ("sweep_T4096", "wide"):
            assert wl.T * wl.k > 4096          # more than one sort chunk
        for seed in (0, 3):
            ids, lr = _route(ml, torch, wl, seed)
            _compare(ml, torch, wl, d, ids, lr)
