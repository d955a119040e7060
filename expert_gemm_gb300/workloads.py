"""Seeded synthetic inputs for the MoE-LoRA layer.

This module draws random numbers and nothing else: it holds none of the
layer's arithmetic (no routing, sorting, GEMM or activation).  Both the CUDA
path and the CPU oracle are fed from here, so that the two see bit-identical
inputs.

Workloads (shapes and distributions follow the configurations the layer is
measured on; the serving workload of the AWS/vLLM post "Efficiently serve
dozens of fine-tuned models with vLLM on Amazon SageMaker AI and Amazon
Bedrock" -- GPT-OSS 20B, 8 adapters of rank 32, 16 concurrent requests of 1600
prompt tokens, section "Implementing multi-LoRA inference for MoE models in
vLLM" and Figure 3 -- is stood in for by synthetic tensors of those shapes):

  tiny        T=64    H=256  I=512   E=8   k=2  L=4  r=8      ids uniform {-1..3}
  decode      T=16    H=2880 I=2880  E=32  k=4  L=8  r=32     ids uniform {0..7}
  prefill     T=25600 H=2880 I=2880  E=32  k=4  L=8  r=32     16 requests x 1600 tokens,
                                                              one uniform adapter per request
  wide        T=4096  H=4096 I=11008 E=8   k=2  L=32 r=32     ids Zipf(1.1), logit bias N(0,1)
  sweep_T{1,16,256,4096}
              T       H=2048 I=768   E=128 k=8  L=64 r{16,64} ids Zipf(1.1) with 10% -1,
                                                              logit bias N(0,0.5)
  dense_decode T=16   H=5120 I=25600 E=1   k=1  L=8  r=32     ids uniform {0..7}
              (multi-LoRA on a dense SwiGLU MLP of a 32B-class model: the single
              "expert" is the MLP; the pages report the same optimisations helping
              dense models, section "Results & Conclusion")

Value recipe: x ~ N(0,1); router logits ~ N(0,1) (fp32, plus the per-expert
bias where the workload has one, added in fp32); W, A, B ~ N(0, 0.02).  Every
bf16 tensor is drawn in fp32 and rounded to bf16 (round to nearest even).

Weight storage (all row-major, "output features x input features", i.e. the
reduction dimension is contiguous):
  W_gu  [E, 2I, H]   rows [0, I) are the gate projection, rows [I, 2I) the up projection
  W_dn  [E, H, I]
  A_gu  [L, E, r_max, H]   LoRA shrink of gate_up (rows >= rank(a) are zero)
  B_gu  [L, E, r_max, 2I]  LoRA expand of gate_up, the r x 2I matrix B of XAB (rows >= rank(a) zero)
  A_dn  [L, E, r_max, I]
  B_dn  [L, E, r_max, H]
Mixed ranks: adapter a has rank 16 when a is even and 64 when a is odd.

Determinism: each tensor, and each slice of it along its leading dimension,
draws from its own PCG64 stream whose key is (seed, tensor number, slice
number).  The result is independent of the order and the number of threads
used to fill it.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

# Tensor numbers: the fixed order of the streams.
_LOGITS, _BIAS, _LORA, _X, _WGU, _WDN, _AGU, _BGU, _ADN, _BDN = range(10)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    k: int
    L: int
    ranks: tuple          # rank of each adapter, len L
    lora_mode: str        # "uniform_with_none" | "uniform" | "per_request" | "zipf" | "zipf_with_none"
    bias_std: float = 0.0
    requests: int = 0     # for per_request
    zipf_s: float = 1.1
    none_frac: float = 0.0
    w_std: float = 0.02
    block_m: int = 0      # token-block size the bench launches with (0 = library's pick)

    @property
    def r_max(self) -> int:
        return max(self.ranks) if self.ranks else 0

    @property
    def P(self) -> int:
        return self.T * self.k


def _sweep(T: int) -> Workload:
    ranks = tuple(16 if a % 2 == 0 else 64 for a in range(64))
    return Workload(f"sweep_T{T}", T, 2048, 768, 128, 8, 64, ranks,
                    "zipf_with_none", bias_std=0.5, none_frac=0.1)


WORKLOADS = {
    "tiny": Workload("tiny", 64, 256, 512, 8, 2, 4, (8,) * 4, "uniform_with_none"),
    "decode": Workload("decode", 16, 2880, 2880, 32, 4, 8, (32,) * 8, "uniform"),
    "prefill": Workload("prefill", 25600, 2880, 2880, 32, 4, 8, (32,) * 8,
                        "per_request", requests=16),
    "wide": Workload("wide", 4096, 4096, 11008, 8, 2, 32, (32,) * 32, "zipf",
                     bias_std=1.0),
    "dense_decode": Workload("dense_decode", 16, 5120, 25600, 1, 1, 8, (32,) * 8, "uniform"),
    "sweep_T1": _sweep(1),
    "sweep_T16": _sweep(16),
    "sweep_T256": _sweep(256),
    "sweep_T4096": _sweep(4096),
}


def custom(name="custom", **kw) -> Workload:
    """A workload with explicit sizes (used for edge cases and small parity runs)."""
    return Workload(name=name, **kw)


def _stream(seed: int, tensor: int, part: int = 0) -> np.random.Generator:
    ss = np.random.SeedSequence(entropy=seed, spawn_key=(tensor, part))
    return np.random.Generator(np.random.PCG64(ss))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _normal_bf16(seed, tensor, shape, std, zero_fn=None):
    """bf16 bits of N(0, std^2) of `shape`; slice i of the leading dim from stream (tensor, i).

    zero_fn(i, slice) may zero parts of slice i in place (rank padding) after drawing.
    """
    out = np.empty(shape, dtype=np.uint16)
    n0 = shape[0]
    inner = tuple(shape[1:])

    def fill(i):
        g = _stream(seed, tensor, i)
        v = g.standard_normal(inner, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        if zero_fn is not None:
            zero_fn(i, v)
        out[i] = f32_to_bf16_bits(v)

    if n0 * int(np.prod(inner, dtype=np.int64)) < (1 << 22):
        for i in range(n0):
            fill(i)
    else:
        with _cf.ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(n0)))
    return out


def _zipf_ids(g: np.random.Generator, n: int, L: int, s: float) -> np.ndarray:
    w = (np.arange(1, L + 1, dtype=np.float64)) ** (-s)
    cdf = np.cumsum(w / w.sum())
    cdf[-1] = 1.0
    u = g.random(n)
    return np.searchsorted(cdf, u, side="right").astype(np.int32)


def make_routing(wl: Workload, seed: int = 0):
    """Router logits (fp32 [T,E], bias included) and adapter ids (int32 [T])."""
    T, E, L = wl.T, wl.E, wl.L
    logits = _stream(seed, _LOGITS).standard_normal((T, E), dtype=np.float32)
    if wl.bias_std:
        bias = _stream(seed, _BIAS).standard_normal(E, dtype=np.float32) * np.float32(wl.bias_std)
        logits = (logits + bias[None, :]).astype(np.float32)
    g = _stream(seed, _LORA)
    if wl.lora_mode == "uniform_with_none":
        lora = g.integers(-1, L, size=T).astype(np.int32)
    elif wl.lora_mode == "uniform":
        lora = g.integers(0, L, size=T).astype(np.int32)
    elif wl.lora_mode == "per_request":
        per = g.integers(0, L, size=wl.requests).astype(np.int32)
        lora = np.repeat(per, T // wl.requests).astype(np.int32)
    elif wl.lora_mode == "zipf":
        lora = _zipf_ids(g, T, L, wl.zipf_s)
    elif wl.lora_mode == "zipf_with_none":
        none = g.random(T) < wl.none_frac
        lora = _zipf_ids(g, T, L, wl.zipf_s)
        lora[none] = -1
    elif wl.lora_mode == "none":
        lora = np.full(T, -1, dtype=np.int32)
    else:
        raise ValueError(wl.lora_mode)
    return np.ascontiguousarray(logits), np.ascontiguousarray(lora)


def make_activations(wl: Workload, seed: int = 0) -> np.ndarray:
    """x: bf16 bits [T, H], N(0,1)."""
    return _normal_bf16(seed, _X, (wl.T, wl.H), 1.0)


def make_weights(wl: Workload, seed: int = 0) -> dict:
    """Expert and adapter weights as bf16 bit arrays (layouts in the module docstring)."""
    E, H, I, L, R = wl.E, wl.H, wl.I, wl.L, wl.r_max
    ranks = np.asarray(wl.ranks, dtype=np.int32)
    s = wl.w_std

    def zero_rows(i, v):      # v: [E, R, K or N] for adapter i -> rows >= rank are zero
        v[:, ranks[i]:, :] = 0

    w = {
        "W_gu": _normal_bf16(seed, _WGU, (E, 2 * I, H), s),
        "W_dn": _normal_bf16(seed, _WDN, (E, H, I), s),
        "A_gu": _normal_bf16(seed, _AGU, (L, E, R, H), s, zero_rows),
        "B_gu": _normal_bf16(seed, _BGU, (L, E, R, 2 * I), s, zero_rows),
        "A_dn": _normal_bf16(seed, _ADN, (L, E, R, I), s, zero_rows),
        "B_dn": _normal_bf16(seed, _BDN, (L, E, R, H), s, zero_rows),
        "ranks": ranks,
    }
    return w


def make_all(wl: Workload, seed: int = 0) -> dict:
    logits, lora = make_routing(wl, seed)
    d = {"logits": logits, "lora_ids": lora, "x": make_activations(wl, seed)}
    d.update(make_weights(wl, seed))
    return d


def get(name: str) -> Workload:
    return WORKLOADS[name]
