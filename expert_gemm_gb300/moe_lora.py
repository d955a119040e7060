"""ctypes binding of libmoe_lora.so (include/moe_lora.h) -- argument marshalling only.

Function names match the C entry points without the `moe_lora_` prefix.  Device
tensors are torch tensors (PyTorch provides device memory and streams); every
step of the layer runs in the library's CUDA kernels.  If the library is missing
the first call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_lora.so")

OK, EINVAL, EALIGN, EWORKSPACE, EUNSUPPORTED, ECUDA, EDEVICE = range(7)
DEV_TIMEOUT = 0x1
MAX_ADAPTERS, MAX_RANK, MAX_EXPERTS, MAX_TOPK = 256, 64, 1024, 32

EXPORTS = ["moe_lora_align_capacity", "moe_lora_workspace_size", "moe_lora_pick_block_m", "moe_lora_route",
           "moe_lora_align", "moe_lora_forward", "moe_lora_layer_workspace_size", "moe_lora_layer_host",
           "moe_lora_status_string", "moe_lora_last_error", "moe_lora_version", "moe_lora_align_static",
           "moe_lora_route_align", "moe_lora_plan_query", "moe_lora_layer_graph_create",
           "moe_lora_layer_graph_run", "moe_lora_layer_graph_destroy", "moe_lora_debug_set_acc_wait_ns",
           "moe_lora_debug_set_shrink_tiles"]
STATIC_SCRATCH_BYTES = 4 << 20


class Dims(C.Structure):
    _fields_ = [("T", C.c_int64), ("H", C.c_int32), ("I", C.c_int32), ("E", C.c_int32), ("k", C.c_int32),
                ("L", C.c_int32), ("r_max", C.c_int32), ("block_m", C.c_int32), ("ranks", C.POINTER(C.c_int32))]


class AlignBuf(C.Structure):
    _fields_ = [("sorted_p", C.c_void_p), ("expert_begin", C.c_void_p), ("block_expert", C.c_void_p),
                ("block_runs", C.c_void_p), ("runs", C.c_void_p), ("totals", C.c_void_p)]


class Plan(C.Structure):
    _fields_ = [("block_m", C.c_int32), ("table_row", C.c_int32), ("weight_streaming", C.c_int32),
                ("ksplit", C.c_int32 * 4), ("k_tile", C.c_int32 * 4), ("stages", C.c_int32 * 4),
                ("launches_route_align", C.c_int32), ("launches_forward", C.c_int32),
                ("shrink_on_cores", C.c_int32), ("shrink_block_diag", C.c_int32)]


GEMMS = ("shrink_gu", "gate_up", "shrink_dn", "down")


class MoeLoraError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"moe_lora status {status}: {msg}")
        self.status = status


_lib = None


def load(path: str = LIB_PATH):
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with expert_gemm_gb300.build.build()")
    lib = C.CDLL(path)
    vp, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
    DP, AP = C.POINTER(Dims), C.POINTER(AlignBuf)
    lib.moe_lora_align_capacity.argtypes = [DP, C.POINTER(i64), C.POINTER(i64), C.POINTER(i64)]
    lib.moe_lora_workspace_size.argtypes = [DP, C.POINTER(sz), C.POINTER(sz)]
    lib.moe_lora_layer_workspace_size.argtypes = [DP, C.POINTER(sz)]
    lib.moe_lora_pick_block_m.argtypes = [i64, i32, i32, i32, i32, i32]
    lib.moe_lora_pick_block_m.restype = i32
    lib.moe_lora_route.argtypes = [vp, i64, i32, i32, vp, vp, vp]
    lib.moe_lora_align.argtypes = [DP, vp, vp, AP, vp, sz, vp]
    lib.moe_lora_align_static.argtypes = [DP, vp, vp, AP, vp]
    lib.moe_lora_route_align.argtypes = [DP, vp, vp, vp, vp, AP, vp, sz, vp]
    lib.moe_lora_plan_query.argtypes = [DP, C.POINTER(Plan)]
    lib.moe_lora_layer_graph_create.argtypes = [DP, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp,
                                                C.POINTER(vp)]
    lib.moe_lora_layer_graph_run.argtypes = [vp, vp, C.POINTER(i64)]
    lib.moe_lora_layer_graph_destroy.argtypes = [vp]
    lib.moe_lora_forward.argtypes = [DP, vp, vp, AP, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp, vp]
    lib.moe_lora_layer_host.argtypes = [DP, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, C.POINTER(i64), vp]
    lib.moe_lora_debug_set_acc_wait_ns.argtypes = [C.c_uint64]
    lib.moe_lora_debug_set_acc_wait_ns.restype = C.c_int
    lib.moe_lora_debug_set_shrink_tiles.argtypes = [C.c_int32]
    lib.moe_lora_debug_set_shrink_tiles.restype = C.c_int
    lib.moe_lora_status_string.restype = C.c_char_p
    lib.moe_lora_status_string.argtypes = [C.c_int]
    lib.moe_lora_last_error.restype = C.c_char_p
    lib.moe_lora_version.restype = C.c_int
    for name in ("moe_lora_align_capacity", "moe_lora_workspace_size", "moe_lora_layer_workspace_size",
                 "moe_lora_route", "moe_lora_align", "moe_lora_forward", "moe_lora_layer_host",
                 "moe_lora_align_static", "moe_lora_route_align", "moe_lora_plan_query",
                 "moe_lora_layer_graph_create", "moe_lora_layer_graph_run", "moe_lora_layer_graph_destroy"):
        getattr(lib, name).restype = C.c_int
    _lib = lib
    return lib


def _check(status: int):
    if status != OK:
        lib = load()
        raise MoeLoraError(status, f"{lib.moe_lora_status_string(status).decode()}: "
                                   f"{lib.moe_lora_last_error().decode()}")


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


@dataclass
class LayerDims:
    """Python mirror of moe_lora_dims (keeps the host ranks array alive)."""
    T: int
    H: int
    I: int
    E: int
    k: int
    L: int
    r_max: int
    block_m: int
    ranks: tuple

    def c(self) -> Dims:
        self._ranks = np.ascontiguousarray(np.asarray(self.ranks, dtype=np.int32).reshape(-1))
        return Dims(self.T, self.H, self.I, self.E, self.k, self.L, self.r_max, self.block_m,
                    self._ranks.ctypes.data_as(C.POINTER(C.c_int32)))


def version() -> int:
    return load().moe_lora_version()


def debug_set_acc_wait_ns(ns: int):
    """Test hook: limit (ns) of the gate_up epilogue's accumulator wait in later forward
    calls (single-CTA kernels); 0 restores the default.  See moe_lora.h."""
    _check(load().moe_lora_debug_set_acc_wait_ns(int(ns)))


def debug_set_shrink_tiles(mode: int):
    """Test hook: tile form of the tcgen05 shrinks of token-tiled blocks in later forward
    calls (0 by shape, 1 block-diagonal, 2 one run per tile).  See moe_lora.h."""
    _check(load().moe_lora_debug_set_shrink_tiles(int(mode)))


def pick_block_m(T: int, k: int, E: int, L: int = 0, H: int = 0, I: int = 0) -> int:
    """The tile table's block_m for T tokens, top-k over E experts, L adapters, experts of
    hidden size H and intermediate size I (0: unknown, the large-expert rule is left out)."""
    return load().moe_lora_pick_block_m(T, k, E, L, H, I)


def plan(d: LayerDims) -> dict:
    """moe_lora_plan_query as a dict (host only)."""
    p = Plan()
    _check(load().moe_lora_plan_query(C.byref(d.c()), C.byref(p)))
    return {"block_m": p.block_m, "table_row": p.table_row, "weight_streaming": bool(p.weight_streaming),
            "ksplit": dict(zip(GEMMS, p.ksplit)), "k_tile": dict(zip(GEMMS, p.k_tile)),
            "stages": dict(zip(GEMMS, p.stages)), "launches_route_align": p.launches_route_align,
            "launches_forward": p.launches_forward, "shrink_on_cores": bool(p.shrink_on_cores),
            "shrink_block_diag": bool(p.shrink_block_diag)}


def align_capacity(d: LayerDims):
    r, b, n = C.c_int64(), C.c_int64(), C.c_int64()
    _check(load().moe_lora_align_capacity(C.byref(d.c()), C.byref(r), C.byref(b), C.byref(n)))
    return r.value, b.value, n.value


def workspace_size(d: LayerDims):
    a, f = C.c_size_t(), C.c_size_t()
    _check(load().moe_lora_workspace_size(C.byref(d.c()), C.byref(a), C.byref(f)))
    return a.value, f.value


def layer_workspace_size(d: LayerDims) -> int:
    n = C.c_size_t()
    _check(load().moe_lora_layer_workspace_size(C.byref(d.c()), C.byref(n)))
    return n.value


def route(logits, k: int, topk_ids, topk_w, stream=None):
    T, E = logits.shape
    _check(load().moe_lora_route(_ptr(logits), T, E, k, _ptr(topk_ids), _ptr(topk_w), _stream(stream)))


def _abuf(bufs: dict) -> AlignBuf:
    return AlignBuf(*[_ptr(bufs[n]) for n in ("sorted_p", "expert_begin", "block_expert", "block_runs", "runs",
                                              "totals")])


def alloc_align(d: LayerDims, device="cuda"):
    """Allocates (with torch) the align output arrays at their capacities."""
    import torch
    rows, blocks, runs = align_capacity(d)
    i32 = dict(dtype=torch.int32, device=device)
    return {"sorted_p": torch.empty(max(rows, 1), **i32), "expert_begin": torch.empty(d.E + 1, **i32),
            "block_expert": torch.empty(max(blocks, 1), **i32), "block_runs": torch.empty(blocks + 1, **i32),
            "runs": torch.empty((max(runs, 1), 4), **i32), "totals": torch.zeros(4, **i32)}


def align(d: LayerDims, topk_ids, lora_ids, bufs: dict, workspace, stream=None):
    _check(load().moe_lora_align(C.byref(d.c()), _ptr(topk_ids), _ptr(lora_ids), C.byref(_abuf(bufs)),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def align_static(d: LayerDims, topk_ids, lora_ids, bufs: dict, stream=None):
    """moe_lora_align with the library's static device scratch instead of a workspace.

    For callers that cannot allocate device memory when they call.  Calls on one
    device share that scratch: do not let them overlap on the GPU.
    """
    _check(load().moe_lora_align_static(C.byref(d.c()), _ptr(topk_ids), _ptr(lora_ids), C.byref(_abuf(bufs)),
                                        _stream(stream)))


def route_align(d: LayerDims, logits, lora_ids, topk_ids, topk_w, bufs: dict, workspace, stream=None):
    """route + align; one launch when T*k <= 4096.  topk_ids, topk_w and bufs are outputs."""
    _check(load().moe_lora_route_align(C.byref(d.c()), _ptr(logits), _ptr(lora_ids), _ptr(topk_ids), _ptr(topk_w),
                                       C.byref(_abuf(bufs)), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream)))


NUM_STAGES = 6
STAGES = ("gather", "shrink_gu", "gate_up", "shrink_dn", "down", "combine")


def forward(d: LayerDims, x, topk_w, bufs: dict, w: dict, out, workspace, dev_status, stream=None,
            stage_events=None):
    """w: device tensors W_gu, W_dn, A_gu, B_gu, A_dn, B_dn (bf16 or int16 bit patterns).

    stage_events: None, or NUM_STAGES + 1 torch.cuda.Event recorded at the stage boundaries.
    """
    ev = None
    if stage_events is not None:
        ev = (C.c_void_p * len(stage_events))(*[e.cuda_event for e in stage_events])
    _check(load().moe_lora_forward(C.byref(d.c()), _ptr(x), _ptr(topk_w), C.byref(_abuf(bufs)),
                                   _ptr(w["W_gu"]), _ptr(w["W_dn"]), _ptr(w.get("A_gu")), _ptr(w.get("B_gu")),
                                   _ptr(w.get("A_dn")), _ptr(w.get("B_dn")), _ptr(out), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _ptr(dev_status),
                                   _stream(stream), ev))


def layer_host(d: LayerDims, logits_host, lora_ids_host, x_host, w: dict, out_host, workspace, stream=None) -> int:
    """Whole layer from host buffers (pinned recommended) to a host output; returns dropped pairs."""
    dropped = C.c_int64()
    _check(load().moe_lora_layer_host(C.byref(d.c()), _ptr(logits_host), _ptr(lora_ids_host), _ptr(x_host),
                                      _ptr(w["W_gu"]), _ptr(w["W_dn"]), _ptr(w.get("A_gu")), _ptr(w.get("B_gu")),
                                      _ptr(w.get("A_dn")), _ptr(w.get("B_dn")), _ptr(out_host), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), C.byref(dropped),
                                      _stream(stream)))
    return dropped.value


class LayerGraph:
    """moe_lora_layer_graph_*: the host-to-host layer captured once, replayed per step.

    Host buffers must be pinned and stay put; each run() reads their current contents.
    """

    def __init__(self, d: LayerDims, logits_host, lora_ids_host, x_host, w: dict, out_host, workspace, stream):
        import torch
        self.status_host = torch.zeros(8, dtype=torch.int32).pin_memory()
        self.stream = stream
        self._keep = (logits_host, lora_ids_host, x_host, out_host, workspace, w)
        h = C.c_void_p()
        _check(load().moe_lora_layer_graph_create(
            C.byref(d.c()), _ptr(logits_host), _ptr(lora_ids_host), _ptr(x_host), _ptr(w["W_gu"]), _ptr(w["W_dn"]),
            _ptr(w.get("A_gu")), _ptr(w.get("B_gu")), _ptr(w.get("A_dn")), _ptr(w.get("B_dn")), _ptr(out_host),
            _ptr(self.status_host), _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream),
            C.byref(h)))
        self.handle = h

    def run(self) -> int:
        """One step; returns the dropped-pair count."""
        dropped = C.c_int64()
        _check(load().moe_lora_layer_graph_run(self.handle, _stream(self.stream), C.byref(dropped)))
        return dropped.value

    def close(self):
        if self.handle:
            _check(load().moe_lora_layer_graph_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Layer:
    """One MoE-LoRA layer with device-resident weights and preallocated scratch.

    `step(logits, lora_ids, x)` runs route+align -> forward on device tensors and
    returns the bf16 output tensor; `step_host(...)` runs the whole layer from host
    buffers through moe_lora_layer_host.
    """

    def __init__(self, dims: LayerDims, weights: dict, device="cuda"):
        import torch
        self.d = dims
        self.device = device
        self.w = weights
        self.bufs = alloc_align(dims, device)
        a, f = workspace_size(dims)
        self.ws_align = torch.empty(max(a, 256), dtype=torch.uint8, device=device)
        self.ws_fwd = torch.empty(max(f, 256), dtype=torch.uint8, device=device)
        self.topk_ids = torch.empty((dims.T, dims.k), dtype=torch.int32, device=device)
        self.topk_w = torch.empty((dims.T, dims.k), dtype=torch.float32, device=device)
        self.out = torch.empty((dims.T, dims.H), dtype=torch.bfloat16, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self._ws_layer = None

    def step(self, logits, lora_ids, x, stream=None, stage_events=None):
        route_align(self.d, logits, lora_ids, self.topk_ids, self.topk_w, self.bufs, self.ws_align, stream)
        forward(self.d, x, self.topk_w, self.bufs, self.w, self.out, self.ws_fwd, self.status, stream,
                stage_events)
        return self.out

    def graph_host(self, logits_host, lora_ids_host, x_host, out_host, stream) -> LayerGraph:
        """The host-to-host layer as a replayable graph on `stream` (pinned host buffers)."""
        import torch
        if self._ws_layer is None:
            self._ws_layer = torch.empty(layer_workspace_size(self.d), dtype=torch.uint8, device=self.device)
        return LayerGraph(self.d, logits_host, lora_ids_host, x_host, self.w, out_host, self._ws_layer, stream)

    def step_host(self, logits_host, lora_ids_host, x_host, out_host, stream=None) -> int:
        import torch
        if self._ws_layer is None:
            self._ws_layer = torch.empty(layer_workspace_size(self.d), dtype=torch.uint8, device=self.device)
        return layer_host(self.d, logits_host, lora_ids_host, x_host, self.w, out_host, self._ws_layer, stream)
