"""Independent references the oracle is pinned against (CPU, test-only).

Each one reaches the oracle's result by a different route: a brute-force sort
instead of a selection loop, batched library matmuls over whole experts
instead of per-pair mat-vecs, LoRA merged into the weights (W + B^T A)
instead of separate shrink and expand, a dense MLP instead of routing.
None of them shares code with the oracle or with the CUDA path.
"""
from __future__ import annotations

import numpy as np
from scipy.special import expit

from expert_gemm_gb300.workloads import bf16_bits_to_f32


def f64(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def route_bruteforce_ids(logits: np.ndarray, k: int) -> np.ndarray:
    """Experts ranked by descending logit, lower index first on ties (Python sort)."""
    T, E = logits.shape
    out = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))
        out[t] = order[:k]
    return out


def align_bruteforce(topk_ids, lora_ids, E, L, BM):
    """The align layout built with sorted() on key tuples and list slicing."""
    topk_ids = np.asarray(topk_ids)
    T, k = topk_ids.shape
    P = T * k
    valid, dropped = [], 0
    for p in range(P):
        e, a = int(topk_ids.flat[p]), int(lora_ids[p // k])
        if 0 <= e < E and -1 <= a < L:
            valid.append((e, a, p))
        else:
            dropped += 1
    valid.sort()
    rows, expert_begin, block_expert = [], [], []
    for e in range(E):
        expert_begin.append(len(rows))
        mine = [p for (ee, a, p) in valid if ee == e]
        pad = (-len(mine)) % BM
        rows += mine + [P] * pad
        block_expert += [e] * ((len(mine) + pad) // BM)
    expert_begin.append(len(rows))
    runs, block_runs = [], []
    for b in range(len(rows) // BM):
        block_runs.append(len(runs))
        seg = rows[b * BM:(b + 1) * BM]
        adap = [None if p == P else int(lora_ids[p // k]) for p in seg]
        i = 0
        while i < BM:
            if adap[i] is None:
                i += 1
                continue
            j = i
            while j < BM and adap[j] == adap[i]:
                j += 1
            if adap[i] >= 0:
                runs.append([b, adap[i], b * BM + i, b * BM + j])
            i = j
    block_runs.append(len(runs))
    return {
        "sorted_p": np.array(rows, dtype=np.int32),
        "expert_begin": np.array(expert_begin, dtype=np.int32),
        "block_expert": np.array(block_expert, dtype=np.int32),
        "block_runs": np.array(block_runs, dtype=np.int32),
        "runs": np.array(runs, dtype=np.int32).reshape(-1, 4),
        "num_rows": len(rows), "num_blocks": len(rows) // BM, "num_runs": len(runs),
        "num_dropped": dropped,
    }


def silu(z):
    return z * expit(z)


def moe_base_batched(x_bits, topk_ids, topk_w, W_gu_bits, W_dn_bits):
    """LoRA-free MoE: every expert applied to ALL tokens by np.matmul, then gathered."""
    X = f64(x_bits)
    Wg, Wd = f64(W_gu_bits), f64(W_dn_bits)
    E, I2, H = Wg.shape
    I = I2 // 2
    T, k = topk_ids.shape
    out = np.zeros((T, H))
    for e in range(E):
        G = X @ Wg[e].T
        D = (silu(G[:, :I]) * G[:, I:]) @ Wd[e].T
        for j in range(k):
            sel = topk_ids[:, j] == e
            out[sel] += topk_w[sel, j, None].astype(np.float64) * D[sel]
    return out


def moe_merged(x_bits, topk_ids, topk_w, lora_ids, w):
    """MoE with each adapter merged into its expert's weights: W' = W + B[:r, :]^T A[:r, :]."""
    X = f64(x_bits)
    Wg, Wd = f64(w["W_gu"]), f64(w["W_dn"])
    Ag, Bg, Ad, Bd = f64(w["A_gu"]), f64(w["B_gu"]), f64(w["A_dn"]), f64(w["B_dn"])
    ranks = w["ranks"]
    E, I2, H = Wg.shape
    I = I2 // 2
    T, k = topk_ids.shape
    out = np.zeros((T, H))
    for t in range(T):
        a = int(lora_ids[t])
        for j in range(k):
            e = int(topk_ids[t, j])
            if not (0 <= e < E):
                continue
            Mg, Md = Wg[e], Wd[e]
            if a >= 0:
                r = int(ranks[a])
                Mg = Mg + Bg[a, e][:r, :].T @ Ag[a, e][:r, :]
                Md = Md + Bd[a, e][:r, :].T @ Ad[a, e][:r, :]
            g = Mg @ X[t]
            d = Md @ (silu(g[:I]) * g[I:])
            out[t] += float(topk_w[t, j]) * d
    return out


def dense_swiglu(x_bits, Wg_bits, Wd_bits):
    """One dense SwiGLU MLP over all tokens: (silu(X Wg^T) * (X Wu^T)) Wd^T."""
    X = f64(x_bits)
    Wg, Wd = f64(Wg_bits), f64(Wd_bits)
    I = Wg.shape[0] // 2
    G = np.matmul(X, Wg.T)
    return np.matmul(silu(G[:, :I]) * G[:, I:], Wd.T)
