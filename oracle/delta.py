"""SSE on a gated delta-rule transition -- TEST INFRASTRUCTURE (float64, numpy).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline
may use this module; nothing on the CUDA side shares code with it.

What it computes.  The close-reading notes of "Scaling Linear Attention with
Sparse State Expansion" name Gated DeltaNet's structured transition (section
2.1, eq. 6) as the alternative to GLA's diagonal decay and list the
combination as future work (section 6); the "动态线性注意力" page gives the
DeltaNet update (section 2.1, eq. 4).  With the states S (c x d, rows indexed
by the key, o = q S) and the SSE router of eqs. 9-10, per token t and head h:

    e_t = softmax(l_t) over N,  T_t = top-k of l_t (ties -> lower index)
    for i in T_t:   S_i <- alpha_t (I - e_t[i] beta_t k_t^T k_t) S_i + e_t[i] beta_t k_t^T v_t
    i not in T_t:   S_i unchanged
    shared:         S_N <- alpha_t (I - beta_t ks_t^T ks_t) S_N + beta_t ks_t^T v_t
    o_t = sum_{i in T_t} e_t[i] (scale q_t) S_i + (scale qs_t) S_N

alpha_t = exp(log_alpha_t) is GDN's scalar gate and beta_t its writing
strength, one of each per (token, head); the router weight e_t[i] scales the
write exactly as in eq. 13 (the delta write beta k^T (v - k S) is the whole
write, so e scales beta); keys are normalised by the caller.  The readings
are listed in the design notes of this repository.

Parity status: pinned by ``tests/test_oracle_delta.py`` (beta = 0 decay-only
closed form, exact retrieval of v at q = k with beta = 1, the product form
of the transition matrices, k = N with equal logits against a single
DeltaNet run, untouched unselected states, planted mistakes).
"""
from __future__ import annotations

import numpy as np

from . import to_f64


def _softmax(x):
    z = np.exp(x - x.max())
    return z / z.sum()


def _topk(l, k):
    return np.argsort(-l, kind="stable")[:k]


def _step(S, e_sel, sel, a, b, q, k, v, qs, ks, use_shared, scale, N):
    """One token on the states S [P, c, d] in place; returns o (d)."""
    for i, e in zip(sel, e_sel):
        # alpha (I - e beta k^T k) S + e beta k^T v
        S[i] = a * (S[i] - e * b * np.outer(k, k @ S[i])) + e * b * np.outer(k, v)
    if use_shared:
        S[N] = a * (S[N] - b * np.outer(ks, ks @ S[N])) + b * np.outer(ks, v)
    o = sum(e * scale * (q @ S[i]) for i, e in zip(sel, e_sel))
    if use_shared:
        o = o + scale * (qs @ S[N])
    return o


def delta_forward(q, k, v, log_alpha, beta, logits, cu_seqlens, *, top_k: int, use_shared: int = 1,
                  scale: float = 1.0, q_shared=None, k_shared=None, initial_state=None) -> dict:
    """Arrays: q, k [T, H, c]; v [T, H, d]; log_alpha, beta [T, H];
    logits [T, H, N]; states [S, H, P, c, d].  Returns out, final_state,
    topk_idx, topk_w."""
    Q, K, V, LA, B, L = (to_f64(x) for x in (q, k, v, log_alpha, beta, logits))
    QS = Q if q_shared is None else to_f64(q_shared)
    KS = K if k_shared is None else to_f64(k_shared)
    T, H, c = Q.shape
    d = V.shape[2]
    N = L.shape[2]
    P = N + (1 if use_shared else 0)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    Sn = len(cu) - 1
    out = np.zeros((T, H, d))
    fin = np.zeros((Sn, H, P, c, d))
    idx = np.zeros((T, H, top_k), dtype=np.int32)
    wts = np.zeros((T, H, top_k))
    for b in range(Sn):
        for h in range(H):
            S = np.zeros((P, c, d)) if initial_state is None else to_f64(initial_state[b, h]).copy()
            for t in range(int(cu[b]), int(cu[b + 1])):
                e = _softmax(L[t, h])
                sel = _topk(L[t, h], top_k)
                idx[t, h] = sel
                wts[t, h] = e[sel]
                out[t, h] = _step(S, e[sel], sel, np.exp(LA[t, h]), B[t, h], Q[t, h], K[t, h], V[t, h],
                                  QS[t, h], KS[t, h], use_shared, scale, N)
            fin[b, h] = S
    return {"out": out, "final_state": fin, "topk_idx": idx, "topk_w": wts}


def delta_decode_step(state, q, k, v, log_alpha, beta, logits, *, top_k: int, use_shared: int = 1,
                      scale: float = 1.0, q_shared=None, k_shared=None) -> dict:
    """One decode step; ``state`` [B, H, P, c, d] float64 is updated in place."""
    Q, K, V, LA, Bt, L = (to_f64(x) for x in (q, k, v, log_alpha, beta, logits))
    QS = Q if q_shared is None else to_f64(q_shared)
    KS = K if k_shared is None else to_f64(k_shared)
    Bn, H, c = Q.shape
    d = V.shape[2]
    N = L.shape[2]
    out = np.zeros((Bn, H, d))
    idx = np.zeros((Bn, H, top_k), dtype=np.int32)
    wts = np.zeros((Bn, H, top_k))
    for b in range(Bn):
        for h in range(H):
            e = _softmax(L[b, h])
            sel = _topk(L[b, h], top_k)
            idx[b, h] = sel
            wts[b, h] = e[sel]
            out[b, h] = _step(state[b, h], e[sel], sel, np.exp(LA[b, h]), Bt[b, h], Q[b, h], K[b, h], V[b, h],
                              QS[b, h], KS[b, h], use_shared, scale, N)
    return {"out": out, "topk_idx": idx, "topk_w": wts}
