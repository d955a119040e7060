"""Shared helpers of the GPU parity tests: upload seeded inputs, run the CUDA path
through the C ABI, and compare with the fp64 oracle."""
from __future__ import annotations

import functools

import numpy as np

from expert_gemm_gb300 import workloads as W

TOL = 2e-2   # max relative error of the layer output, fp32 accumulation, bf16 I/O


def parity_error(y: np.ndarray, ref: np.ndarray):
    """max_i |y_i - ref_i| / max(|ref_i|, rms(ref)) and the norm-wise relative error."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    floor = max(rms, 1e-30)
    elem = float(np.max(np.abs(y - ref) / np.maximum(np.abs(ref), floor))) if ref.size else 0.0
    norm = float(np.linalg.norm(y - ref) / max(np.linalg.norm(ref), 1e-30)) if ref.size else 0.0
    return elem, norm


@functools.lru_cache(maxsize=2)
def weights_for(key):
    """Weights depend only on the layer shapes (not on T); cache them across T values."""
    H, I, E, L, ranks, seed = key
    wl = W.custom(name="w", T=1, H=H, I=I, E=E, k=1, L=L, ranks=ranks, lora_mode="none")
    return W.make_weights(wl, seed)


def inputs(wl: W.Workload, seed: int = 0):
    logits, lora = W.make_routing(wl, seed)
    x = W.make_activations(wl, seed)
    w = weights_for((wl.H, wl.I, wl.E, wl.L, tuple(wl.ranks), seed))
    return logits, lora, x, w


def to_dev(arr: np.ndarray, torch):
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr)).cuda()


_dev_cache = {}


def dev_weights(w: dict, torch):
    key = id(w)
    if key not in _dev_cache:
        _dev_cache.clear()
        torch.cuda.empty_cache()
        _dev_cache[key] = {n: to_dev(w[n], torch) for n in ("W_gu", "W_dn", "A_gu", "B_gu", "A_dn", "B_dn")}
    return _dev_cache[key]


def dims_of(wl: W.Workload, block_m: int, ml, T=None):
    return ml.LayerDims(T=wl.T if T is None else T, H=wl.H, I=wl.I, E=wl.E, k=wl.k, L=wl.L, r_max=wl.r_max,
                        block_m=block_m, ranks=tuple(wl.ranks))


def align_to_numpy(bufs: dict):
    tot = bufs["totals"].cpu().numpy()
    rows, nb, nr, dropped = (int(v) for v in tot)
    return {"sorted_p": bufs["sorted_p"][:rows].cpu().numpy(), "expert_begin": bufs["expert_begin"].cpu().numpy(),
            "block_expert": bufs["block_expert"][:nb].cpu().numpy(),
            "block_runs": bufs["block_runs"][:nb + 1].cpu().numpy(), "runs": bufs["runs"][:nr].cpu().numpy(),
            "num_rows": rows, "num_blocks": nb, "num_runs": nr, "num_dropped": dropped}


def assert_align_equal(got: dict, ref: dict):
    for k in ("num_rows", "num_blocks", "num_runs", "num_dropped"):
        assert got[k] == ref[k], (k, got[k], ref[k])
    for k in ("sorted_p", "expert_begin", "block_expert", "block_runs", "runs"):
        a, b = np.asarray(got[k]).reshape(-1), np.asarray(ref[k]).reshape(-1)
        assert a.shape == b.shape and np.array_equal(a, b), k


# ------------------------------------------------------------------ guards --
# compute-sanitizer is not available here, so out-of-bounds writes are caught with
# canary bytes: each output and scratch buffer of a call is a slice of a larger
# allocation whose head and tail hold a fixed pattern, checked after the call.
GUARD_BYTES = 4096        # keeps every slice 4 KB-aligned (TMA wants 16 bytes)
GUARD_PATTERN = 0xA5


class Guarded:
    """Device buffers carved out of canary-padded allocations."""

    def __init__(self, torch):
        self.torch = torch
        self.bufs = []

    def empty(self, shape, dtype):
        torch = self.torch
        n = int(np.prod(shape)) * torch.empty(0, dtype=dtype).element_size()
        raw = torch.full((n + 2 * GUARD_BYTES,), GUARD_PATTERN, dtype=torch.uint8, device="cuda")
        self.bufs.append((raw, n))
        return raw[GUARD_BYTES:GUARD_BYTES + n].view(dtype).view(shape)

    def guard_layer(self, layer):
        """Swaps a Layer's output, align arrays and workspaces for guarded ones."""
        layer.out = self.empty(tuple(layer.out.shape), layer.out.dtype)
        layer.ws_align = self.empty(tuple(layer.ws_align.shape), layer.ws_align.dtype)
        layer.ws_fwd = self.empty(tuple(layer.ws_fwd.shape), layer.ws_fwd.dtype)
        layer.bufs = {k: self.empty(tuple(v.shape), v.dtype) for k, v in layer.bufs.items()}
        layer.topk_ids = self.empty(tuple(layer.topk_ids.shape), layer.topk_ids.dtype)
        layer.topk_w = self.empty(tuple(layer.topk_w.shape), layer.topk_w.dtype)
        return layer

    def check(self):
        for raw, n in self.bufs:
            head = raw[:GUARD_BYTES]
            tail = raw[GUARD_BYTES + n:]
            assert bool((head == GUARD_PATTERN).all()), f"canary before a {n}-byte buffer overwritten"
            assert bool((tail == GUARD_PATTERN).all()), f"canary after a {n}-byte buffer overwritten"

