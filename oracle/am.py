"""fp64 oracle of Attention Matching (AM): a bias beta and compact values V_C fitted on the
token-eviction survivors.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU legs of
``bench.py`` may import this module.  It shares no code with the CUDA library and never
imports it.  Plain numpy in fp64; every step is written out in the order the method takes it.

Source: "Practical Online KV Cache Compaction for LLM Agents: An Empirical Study" (agifrontier
tutorial page), section on the two families of sequence-level compaction.  AM first keeps the
top-m keys K_C of the token-eviction score, then solves by an optimisation for an additive
attention bias beta (one value per kept key) and a rebuilt compact value matrix V_C so that the
compacted attention reproduces the full one on the proxy queries Q:

    min_beta || exp(Q K_C^T + beta) 1_m - exp(Q K^T) 1_n ||_2^2                      (mass fit)
    min_V_C  || A_hat(Q; K_C, beta, V_C) - A(Q; K, V) ||_F^2                          (value fit)

with A(Q; K, V) = softmax(Q K^T) V the attention output and A_hat the same with logits
Q K_C^T + beta over the kept keys and values V_C.

Readings where the page leaves a step open (each restated in the design notes):

* logits carry the attention scale, L = scale * Q K^T, as in the token-eviction score;
* w = exp(beta) >= 0 turns the mass fit into non-negative least squares in w; beta_j = ln w_j,
  and w_j = 0 (beta_j = -inf) masks the key;
* both fits are invariant to one common shift of all logits of a unit; the shift used is the
  largest row log-mass c = max_i LSE_i, so that E = exp(L_C - c) <= 1 and s = exp(LSE - c) <= 1;
* "an optimisation algorithm" is read as cyclic coordinate descent on the normal equations,
  T sweeps over the kept keys in ascending position order, started from token eviction's own
  answer (w = 1, i.e. beta = 0, and V_C = the kept keys' values): projected onto w >= 0 for the
  mass fit, unconstrained for the value fit; the value fit uses the fitted beta.  As T grows
  the iterates reach the non-negative and the ordinary least-squares minimisers (pinned in
  ``tests/test_oracle_am.py`` against brute force and library solvers);
* a key whose column is all zero (every exp underflowed, or w_j = 0 in the value fit) is left
  where it starts.

The iteration is the plain one: every coordinate whose step is non-zero takes it.  Whatever an
implementation in lower precision does to keep rounding out of its steps is its own choice and
is judged by the residuals it reaches, not written into this oracle.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def logits(Q: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """L = scale * Q K^T (R x n)."""
    return scale * (np.asarray(Q, np.float64) @ np.asarray(K, np.float64).T)


def targets(Q, K, V, scale):
    """(lse [R], Y [R][d]) of the full attention: LSE_i = ln sum_j exp(L_ij) and
    Y = softmax(L) V = A(Q; K, V)."""
    L = logits(Q, K, scale)
    mx = L.max(axis=1)
    e = np.exp(L - mx[:, None])
    tot = e.sum(axis=1)
    lse = mx + np.log(tot)
    Y = (e / tot[:, None]) @ np.asarray(V, np.float64)
    return lse, Y


def mass_fit(E: np.ndarray, s: np.ndarray, sweeps: int, w0=None) -> np.ndarray:
    """Projected cyclic coordinate descent on min_{w >= 0} ||E w - s||^2, from w0 (default 1).

    Normal equations G = E^T E, b = E^T s, gradient g = G w - b; coordinate j moves to the
    minimiser of the objective along e_j, clipped at 0: w_j <- max(0, w_j - g_j / G_jj)."""
    E = np.asarray(E, np.float64)
    m = E.shape[1]
    G = E.T @ E
    b = E.T @ np.asarray(s, np.float64)
    w = np.ones(m) if w0 is None else np.array(w0, np.float64)
    g = G @ w - b
    for _ in range(sweeps):
        for j in range(m):
            if not G[j, j] > 0.0:
                continue
            nw = max(0.0, w[j] - g[j] / G[j, j])
            dl = nw - w[j]
            if dl != 0.0:
                g += dl * G[:, j]
                w[j] = nw
    return w


def value_fit(Ph: np.ndarray, Y: np.ndarray, X0: np.ndarray, sweeps: int) -> np.ndarray:
    """Cyclic coordinate descent on min_X ||Ph X - Y||_F^2 from X0, one key (row of X) at a
    time: H = Ph^T Ph, B = Ph^T Y, gradient Gv = H X - B; row j of X moves by -Gv_j / H_jj."""
    Ph = np.asarray(Ph, np.float64)
    Y = np.asarray(Y, np.float64)
    m = Ph.shape[1]
    H = Ph.T @ Ph
    B = Ph.T @ Y
    X = np.array(X0, np.float64)
    Gv = H @ X - B
    for _ in range(sweeps):
        for j in range(m):
            if not H[j, j] > 0.0:
                continue
            dl = -Gv[j] / H[j, j]
            X[j] += dl
            Gv += np.outer(H[:, j], dl)
    return X


def compact_probs(E: np.ndarray, w: np.ndarray) -> np.ndarray:
    """Ph = softmax(L_C + beta) over the kept keys = rows of E diag(w), normalised (a row with no
    mass stays zero)."""
    Ew = np.asarray(E, np.float64) * np.asarray(w, np.float64)[None, :]
    z = Ew.sum(axis=1)
    out = np.zeros_like(Ew)
    nz = z > 0
    out[nz] = Ew[nz] / z[nz, None]
    return out


def beta_of(w: np.ndarray) -> np.ndarray:
    """beta = ln w, -inf where w = 0."""
    w = np.asarray(w, np.float64)
    out = np.full(w.shape, -np.inf)
    pos = w > 0
    out[pos] = np.log(w[pos])
    return out


def unit(Q, K, V, keep, scale, sweeps):
    """AM on one (layer, head, sequence): returns a dict with the fitted w, beta, V_C (as vc),
    the shifted problem (E, s, Y, c) the objectives are measured on, and the value fit's start
    (x0, the kept keys' values)."""
    keep = np.asarray(keep, np.int64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    lse, Y = targets(Q, K, V, scale)
    c = lse.max()
    s = np.exp(lse - c)
    E = np.exp(logits(Q, K[keep], scale) - c)
    w = mass_fit(E, s, sweeps)
    vc = value_fit(compact_probs(E, w), Y, V[keep], sweeps)
    return {"w": w, "beta": beta_of(w), "vc": vc, "E": E, "s": s, "Y": Y, "c": c, "lse": lse,
            "x0": V[keep]}


def mass_objective(E, s, w) -> float:
    """||E w - s||^2 (the mass fit in shifted units, exp(-2c) times the page's form)."""
    r = np.asarray(E, np.float64) @ np.asarray(w, np.float64) - np.asarray(s, np.float64)
    return float(r @ r)


def value_objective(E, Y, w, X) -> float:
    """||Ph(w) X - Y||_F^2 with Ph the compact attention of the kept keys under bias ln w."""
    r = compact_probs(E, w) @ np.asarray(X, np.float64) - np.asarray(Y, np.float64)
    return float((r * r).sum())


def gather(pool_bits, block_table, layer, head, b, s0, s1):
    """Rows [s1 - s0][d] (fp64) of slots [s0, s1) of sequence b from a bf16 pool
    [L][num_pages][H][P][d] given as uint16 bits."""
    P = pool_bits.shape[3]
    slots = np.arange(s0, s1)
    pages = np.asarray(block_table)[b][slots // P]
    return bf16_to_f64(pool_bits[layer, pages, head, slots % P])


def cache(k_bits, v_bits, q_bits, block_table, seg_start, seg_end, keep, m, scale, sweeps):
    """AM on every unit of a paged cache.

    k_bits, v_bits: uint16 [L][num_pages][H][P][d]; q_bits: uint16 [B][L][H][R][d]; keep int32
    [L][H][Mtot] (segment-relative ascending positions, sequence b at offset sum of the earlier
    min(m, n)).  Returns (w [L][H][Mtot], vc [L][H][Mtot][d], units) where units[(b, l, h)] is
    the dict of ``unit``."""
    L, _, H, _, d = k_bits.shape
    B = len(seg_start)
    n = [int(e) - int(s) for s, e in zip(seg_start, seg_end)]
    mm = [min(int(a), x) for a, x in zip(m, n)]
    Mtot = int(sum(mm))
    w_all = np.zeros((L, H, Mtot))
    vc_all = np.zeros((L, H, Mtot, d))
    units = {}
    off = 0
    for b in range(B):
        if mm[b] > 0:
            for l in range(L):
                for h in range(H):
                    K = gather(k_bits, block_table, l, h, b, seg_start[b], seg_end[b])
                    V = gather(v_bits, block_table, l, h, b, seg_start[b], seg_end[b])
                    Q = bf16_to_f64(q_bits[b, l, h])
                    kp = np.asarray(keep[l, h, off:off + mm[b]], np.int64)
                    u = unit(Q, K, V, kp, scale, sweeps)
                    w_all[l, h, off:off + mm[b]] = u["w"]
                    vc_all[l, h, off:off + mm[b]] = u["vc"]
                    units[(b, l, h)] = u
        off += mm[b]
    return w_all, vc_all, units
