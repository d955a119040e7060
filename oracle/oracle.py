"""Python front end of the fp64 CPU oracle (moe_lora_oracle.c).

TEST INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The product path never
imports this module.  It shares no code with the CUDA library.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_lora_oracle.c")
LIB = os.path.join(HERE, "libmoe_lora_oracle.so")

_lib = None


def build(force: bool = False, src: str = SRC, out: str = LIB) -> str:
    """Compile the oracle with gcc + OpenMP (plain C, no target-specific flags)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                        src, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, out)
    return out


def _ptr(a, ctype):
    return a.ctypes.data_as(C.POINTER(ctype))


I32P, I64P, F32P, F64P, U16P = (C.POINTER(C.c_int32), C.POINTER(C.c_int64), C.POINTER(C.c_float),
                                C.POINTER(C.c_double), C.POINTER(C.c_uint16))


def load(path: str | None = None):
    """Load (building if needed) the oracle library; `path` loads a specific build."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = C.CDLL(path or build())
    lib.oracle_route.argtypes = [F32P, C.c_int64, C.c_int32, C.c_int32, I32P, F64P]
    lib.oracle_route.restype = None
    lib.oracle_align.argtypes = [C.c_int64, C.c_int32, C.c_int32, C.c_int32, C.c_int32,
                                 I32P, I32P, I32P, C.c_int64, I32P, I32P, I32P, C.c_int64,
                                 I32P, C.c_int64, I64P]
    lib.oracle_align.restype = C.c_int
    lib.oracle_forward.argtypes = [C.c_int64] + [C.c_int32] * 6 + [I32P, U16P, I32P, F32P, I32P] + \
        [U16P] * 6 + [I64P, C.c_int64, F64P, I64P]
    lib.oracle_forward.restype = None
    lib.oracle_set_threads.argtypes = [C.c_int32]
    lib.oracle_set_threads.restype = C.c_int32
    if path is None:
        _lib = lib
    return lib


class Oracle:
    """Callable wrapper around one loaded oracle library (default: the committed source)."""

    def __init__(self, path: str | None = None):
        self.lib = load(path)

    def set_threads(self, n: int) -> int:
        """OpenMP threads of later calls from this thread (n <= 0: one per processor)."""
        return int(self.lib.oracle_set_threads(int(n)))

    def route(self, logits: np.ndarray, k: int):
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        T, E = logits.shape
        ids = np.empty((T, k), dtype=np.int32)
        w = np.empty((T, k), dtype=np.float64)
        self.lib.oracle_route(_ptr(logits, C.c_float), T, E, k, _ptr(ids, C.c_int32), _ptr(w, C.c_double))
        return ids, w

    @staticmethod
    def capacity(T: int, E: int, k: int, L: int, BM: int):
        """Upper bounds on rows, blocks and runs of the align layout."""
        P = T * k
        rows = P + min(E, P) * (BM - 1)
        rows = (rows + BM - 1) // BM * BM
        blocks = rows // BM
        runs = min(P, blocks + E * max(L, 1))
        return rows, blocks, runs

    def align(self, topk_ids: np.ndarray, lora_ids: np.ndarray, E: int, L: int, BM: int):
        topk_ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
        lora_ids = np.ascontiguousarray(lora_ids, dtype=np.int32)
        T, k = topk_ids.shape
        cap_rows, cap_blocks, cap_runs = self.capacity(T, E, k, L, BM)
        sorted_p = np.full(max(cap_rows, 1), -7, dtype=np.int32)
        expert_begin = np.zeros(E + 1, dtype=np.int32)
        block_expert = np.full(max(cap_blocks, 1), -7, dtype=np.int32)
        block_runs = np.full(cap_blocks + 1, -7, dtype=np.int32)
        runs = np.full((max(cap_runs, 1), 4), -7, dtype=np.int32)
        totals = np.zeros(4, dtype=np.int64)
        rc = self.lib.oracle_align(T, E, k, L, BM, _ptr(topk_ids, C.c_int32), _ptr(lora_ids, C.c_int32),
                                   _ptr(sorted_p, C.c_int32), cap_rows, _ptr(expert_begin, C.c_int32),
                                   _ptr(block_expert, C.c_int32), _ptr(block_runs, C.c_int32), cap_blocks,
                                   _ptr(runs, C.c_int32), cap_runs, _ptr(totals, C.c_int64))
        if rc != 0:
            raise RuntimeError("oracle_align: capacity exceeded")
        n_rows, nb, nr, dropped = (int(v) for v in totals)
        return {
            "sorted_p": sorted_p[:n_rows].copy(),
            "expert_begin": expert_begin,
            "block_expert": block_expert[:nb].copy(),
            "block_runs": block_runs[:nb + 1].copy(),
            "runs": runs[:nr].copy(),
            "num_rows": n_rows, "num_blocks": nb, "num_runs": nr, "num_dropped": dropped,
        }

    def forward(self, x, topk_ids, topk_w, lora_ids, w: dict, tokens=None):
        """fp64 layer output [T or len(tokens), H]; weights as bf16 bit arrays (workloads layout)."""
        x = np.ascontiguousarray(x, dtype=np.uint16)
        topk_ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
        topk_w = np.ascontiguousarray(topk_w, dtype=np.float32)
        lora_ids = np.ascontiguousarray(lora_ids, dtype=np.int32)
        T, H = x.shape
        k = topk_ids.shape[1]
        E, I2, _ = w["W_gu"].shape
        I = I2 // 2
        L, _, R, _ = w["A_gu"].shape
        ranks = np.ascontiguousarray(w["ranks"], dtype=np.int32)
        arrs = [np.ascontiguousarray(w[n], dtype=np.uint16) for n in ("W_gu", "W_dn", "A_gu", "B_gu", "A_dn", "B_dn")]
        if tokens is None:
            tok_p, n_out = None, T
        else:
            tokens = np.ascontiguousarray(tokens, dtype=np.int64)
            tok_p, n_out = _ptr(tokens, C.c_int64), len(tokens)
        out = np.zeros((n_out, H), dtype=np.float64)
        dropped = np.zeros(1, dtype=np.int64)
        self.lib.oracle_forward(T, H, I, E, k, L, R, _ptr(ranks, C.c_int32), _ptr(x, C.c_uint16),
                                _ptr(topk_ids, C.c_int32), _ptr(topk_w, C.c_float), _ptr(lora_ids, C.c_int32),
                                *[_ptr(a, C.c_uint16) for a in arrs], tok_p, n_out,
                                _ptr(out, C.c_double), _ptr(dropped, C.c_int64))
        return out

    def layer(self, logits, lora_ids, x, w: dict, k: int, BM: int, tokens=None):
        """route -> align -> forward, as one pass over the layer."""
        ids, tw = self.route(logits, k)
        al = self.align(ids, lora_ids, logits.shape[1], w["A_gu"].shape[0], BM)
        out = self.forward(x, ids, tw.astype(np.float32), lora_ids, w, tokens)
        return ids, tw, al, out
