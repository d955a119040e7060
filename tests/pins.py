"""Pins of the fp64 oracle: each check compares it with something other than itself.

Every pin is a plain function of an oracle instance, so that the same checks run
against the committed oracle (test_oracle_pins.py) and against copies of it with
a planted mistake (test_oracle_mutants.py), where at least one pin must fail.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
from scipy.special import softmax

import independent as ind
from expert_gemm_gb300 import workloads as wlmod
from expert_gemm_gb300.workloads import f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _small_case(seed=3, T=24, H=32, I=40, E=5, k=2, L=3, ranks=(8, 16, 8), lora_mode="uniform_with_none"):
    wl = wlmod.custom(name="pin", T=T, H=H, I=I, E=E, k=k, L=L, ranks=tuple(ranks), lora_mode=lora_mode,
                      w_std=0.2)
    return wl, wlmod.make_all(wl, seed)


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ---------------------------------------------------------------- route -----

def pin_route_bruteforce(o):
    """Top-k ids equal a Python sort on (-logit, index); includes forced ties."""
    g = np.random.default_rng(11)
    for T, E, k in [(40, 8, 2), (17, 32, 4), (9, 128, 8), (5, 6, 6), (3, 3, 1)]:
        logits = g.standard_normal((T, E)).astype(np.float32)
        logits[:, 1] = logits[:, 0]                       # exact tie between experts 0 and 1
        logits[0, :] = 0.5                                # a token whose logits all tie
        ids, w = o.route(logits, k)
        assert np.array_equal(ids, ind.route_bruteforce_ids(logits, k)), (T, E, k)


def pin_route_weights(o):
    """Weights: k=1 gives 1; k=E gives scipy's softmax; w_i/w_j = exp(l_i - l_j); sums are 1."""
    g = np.random.default_rng(12)
    logits = (3 * g.standard_normal((20, 8))).astype(np.float32)
    _, w1 = o.route(logits, 1)
    assert np.all(w1 == 1.0)
    ids, wE = o.route(logits, 8)
    sm = softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(wE, np.take_along_axis(sm, ids, axis=1), rtol=1e-13, atol=0)
    ids, w3 = o.route(logits, 3)
    assert np.allclose(w3.sum(1), 1.0, rtol=0, atol=1e-14)
    l3 = np.take_along_axis(logits.astype(np.float64), ids, axis=1)
    assert np.allclose(w3[:, 0] / w3[:, 1], np.exp(l3[:, 0] - l3[:, 1]), rtol=1e-12)
    assert np.all(np.diff(w3, axis=1) <= 0)


# ---------------------------------------------------------------- align -----

def _align_equal(a, b):
    for key in ("sorted_p", "expert_begin", "block_expert", "block_runs", "runs"):
        if not np.array_equal(np.asarray(a[key]).reshape(-1), np.asarray(b[key]).reshape(-1)):
            return key
    for key in ("num_rows", "num_blocks", "num_runs", "num_dropped"):
        if a[key] != b[key]:
            return key
    return None


def pin_align_exhaustive(o):
    """Every (topk_ids, lora_ids) on tiny sizes, incl. invalid ids, equals the sorted()-based layout."""
    n = 0
    for T, k, E, L, BM in [(1, 2, 3, 2, 2), (2, 1, 3, 2, 2), (2, 2, 2, 1, 3), (3, 1, 2, 2, 1)]:
        e_vals = range(-1, E + 1)
        a_vals = range(-2, L + 1)
        for ids in itertools.product(e_vals, repeat=T * k):
            ids_a = np.array(ids, dtype=np.int32).reshape(T, k)
            for lor in itertools.product(a_vals, repeat=T):
                lor_a = np.array(lor, dtype=np.int32)
                got = o.align(ids_a, lor_a, E, L, BM)
                ref = ind.align_bruteforce(ids_a, lor_a, E, L, BM)
                bad = _align_equal(got, ref)
                assert bad is None, (T, k, E, L, BM, ids, lor, bad)
                n += 1
    assert n > 1000


def pin_align_random(o):
    """Larger random cases equal the sorted()-based layout; invariants of the layout hold."""
    g = np.random.default_rng(13)
    for T, k, E, L, BM in [(50, 4, 8, 5, 16), (64, 2, 8, 4, 8), (33, 8, 16, 3, 4), (200, 2, 4, 2, 128)]:
        ids = g.integers(-1, E + 1, size=(T, k)).astype(np.int32)
        lor = g.integers(-1, L, size=T).astype(np.int32)
        got = o.align(ids, lor, E, L, BM)
        ref = ind.align_bruteforce(ids, lor, E, L, BM)
        assert _align_equal(got, ref) is None
        P = T * k
        sp = got["sorted_p"]
        assert got["num_rows"] % BM == 0
        real = sp[sp != P]
        valid = [p for p in range(P) if 0 <= ids.flat[p] < E]
        assert sorted(real.tolist()) == valid                 # a permutation of the valid pairs
        keys = [(int(ids.flat[p]), int(lor[p // k]), int(p)) for p in real]
        assert keys == sorted(keys)                           # keys non-decreasing
        # runs tile the rows of adapter >= 0 exactly
        covered = np.zeros(len(sp), dtype=int)
        for b, a, s, e in got["runs"]:
            assert b * BM <= s < e <= (b + 1) * BM
            covered[s:e] += 1
            assert all(lor[p // k] == a for p in sp[s:e])
        want = np.array([1 if p != P and lor[p // k] >= 0 else 0 for p in sp])
        assert np.array_equal(covered, want)


def pin_align_golden(o):
    """Hand-derived layouts in tests/golden/hand_align.json."""
    doc = json.load(open(os.path.join(GOLDEN, "hand_align.json")))
    for c in doc["cases"]:
        got = o.align(np.array(c["topk_ids"], dtype=np.int32), np.array(c["lora_ids"], dtype=np.int32),
                      c["E"], c["L"], c["BM"])
        exp = {"sorted_p": c["sorted_p"], "expert_begin": c["expert_begin"], "block_expert": c["block_expert"],
               "block_runs": c["block_runs"], "runs": c["runs"], "num_rows": c["totals"][0],
               "num_blocks": c["totals"][1], "num_runs": c["totals"][2], "num_dropped": c["totals"][3]}
        assert _align_equal(got, exp) is None, c["name"]


# -------------------------------------------------------------- forward -----

def pin_forward_zero_B(o):
    """B = 0 gives exactly the same output as adapter id -1 for every token."""
    wl, d = _small_case()
    ids, w = o.route(d["logits"], wl.k)
    w = w.astype(np.float32)
    wz = dict(d)
    wz["B_gu"] = np.zeros_like(d["B_gu"])
    wz["B_dn"] = np.zeros_like(d["B_dn"])
    a = o.forward(d["x"], ids, w, d["lora_ids"], wz)
    b = o.forward(d["x"], ids, w, np.full(wl.T, -1, np.int32), d)
    assert np.array_equal(a, b)


def pin_forward_base_matmul(o):
    """Adapter id -1 everywhere equals whole-expert np.matmul MoE (relative 1e-12)."""
    wl, d = _small_case(seed=4)
    ids, w = o.route(d["logits"], wl.k)
    w = w.astype(np.float32)
    got = o.forward(d["x"], ids, w, np.full(wl.T, -1, np.int32), d)
    ref = ind.moe_base_batched(d["x"], ids, w, d["W_gu"], d["W_dn"])
    assert _rel(got, ref) < 1e-12


def pin_forward_merged(o):
    """Shrink/expand equals merged weights W + B^T A per (adapter, expert), mixed ranks (relative 1e-10)."""
    wl, d = _small_case(seed=5)
    ids, w = o.route(d["logits"], wl.k)
    w = w.astype(np.float32)
    got = o.forward(d["x"], ids, w, d["lora_ids"], d)
    ref = ind.moe_merged(d["x"], ids, w, d["lora_ids"], d)
    assert (d["lora_ids"] >= 0).any() and (d["lora_ids"] < 0).any()
    assert _rel(got, ref) < 1e-10


def pin_forward_dense(o):
    """E=1, k=1 reduces to one dense SwiGLU MLP (np.matmul), relative 1e-12."""
    wl, d = _small_case(seed=6, E=1, k=1, L=1, ranks=(8,), lora_mode="none")
    ids, w = o.route(d["logits"], 1)
    assert np.all(ids == 0) and np.all(w == 1.0)
    got = o.forward(d["x"], ids, w.astype(np.float32), d["lora_ids"], d)
    ref = ind.dense_swiglu(d["x"], d["W_gu"][0], d["W_dn"][0])
    assert _rel(got, ref) < 1e-12


def pin_forward_dropped(o):
    """Pairs with an invalid expert or adapter contribute nothing; tokens without pairs give 0."""
    wl, d = _small_case(seed=7)
    ids, w = o.route(d["logits"], wl.k)
    w = w.astype(np.float32)
    ids2 = ids.copy()
    ids2[0, :] = wl.E            # token 0: all pairs invalid
    ids2[1, 1] = -1              # token 1: second pair invalid
    lor = d["lora_ids"].copy()
    lor[2] = wl.L                # token 2: invalid adapter -> all its pairs dropped
    out = o.forward(d["x"], ids2, w, lor, d)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    w1 = w.copy()
    w1[1, 1] = 0.0
    ref1 = o.forward(d["x"], ids, w1, lor, d)[1]
    assert _rel(out[1], ref1) < 1e-14


def pin_forward_rank_padding_unread(o):
    """Storage beyond each adapter's rank is not part of the layer: garbage there changes nothing."""
    wl, d = _small_case(seed=8)
    ids, w = o.route(d["logits"], wl.k)
    w = w.astype(np.float32)
    ref = o.forward(d["x"], ids, w, d["lora_ids"], d)
    g = np.random.default_rng(9)
    dd = dict(d)
    for name, axis in (("A_gu", 2), ("A_dn", 2), ("B_gu", 2), ("B_dn", 2)):
        arr = d[name].copy()
        for a, r in enumerate(d["ranks"]):
            sl = [a, slice(None), slice(None), slice(None)]
            sl[axis] = slice(int(r), None)
            junk = g.standard_normal(arr[tuple(sl)].shape).astype(np.float32)
            arr[tuple(sl)] = f32_to_bf16_bits(junk)
        dd[name] = arr
    assert np.array_equal(o.forward(d["x"], ids, w, d["lora_ids"], dd), ref)


def _eval(expr):
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))        # noqa: E731
    silu = lambda z: z * sig(z)                        # noqa: E731
    return float(eval(expr, {"sig": sig, "silu": silu, "__builtins__": {}}))


def pin_forward_golden(o):
    """Hand-derived single-token layers in tests/golden/hand_layer.json (closed forms)."""
    doc = json.load(open(os.path.join(GOLDEN, "hand_layer.json")))
    cm = doc["common"]
    bits = lambda v: f32_to_bf16_bits(np.array(v, dtype=np.float32))   # noqa: E731
    wts = {n: bits(cm[n]) for n in ("W_gu", "W_dn", "A_gu", "B_gu", "A_dn", "B_dn")}
    wts["ranks"] = np.array(cm["ranks"], dtype=np.int32)
    for c in doc["cases"]:
        logits = np.array(c["logits"], dtype=np.float32)
        ids, w = o.route(logits, cm["k"])
        assert np.array_equal(ids, np.array(c["topk_ids"])), c["name"]
        w_exp = np.array([[_eval(s) for s in row] for row in c["topk_w"]])
        assert np.allclose(w, w_exp, rtol=1e-15, atol=0), c["name"]
        out = o.forward(bits(cm["x"]), ids, w.astype(np.float32), np.array(c["lora_ids"], np.int32), wts)
        o_exp = np.array([[_eval(s) for s in row] for row in c["out"]])
        # weights enter the layer in fp32: allow the fp32 rounding of w only
        assert np.allclose(out, o_exp, rtol=2e-7, atol=1e-12), (c["name"], out, o_exp)


ALL_PINS = [pin_route_bruteforce, pin_route_weights, pin_align_exhaustive, pin_align_random, pin_align_golden,
            pin_forward_zero_B, pin_forward_base_matmul, pin_forward_merged, pin_forward_dense,
            pin_forward_dropped, pin_forward_rank_padding_unread, pin_forward_golden]
