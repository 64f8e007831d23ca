"""Backward of the SSE layer -- TEST INFRASTRUCTURE (float64, numpy).

Only ``tests/`` may use this module; nothing on the CUDA side shares code with
it.  Small cases only (token-by-token loops with every state kept).

What it differentiates: the forward of "Scaling Linear Attention with Sparse
State Expansion" (close-reading notes, section 2.3, eqs. 9-14, plus the
always-on shared partition of section 2.5), per sequence and head:

    e_t = softmax(l_t) over N,  T_t = top-k of l_t (ties -> lower index)
    S_i <- diag(a_t) S_i + e_t[i] k_t^T v_t   for i in T_t,  a_t = exp(g_t)
    S_N <- diag(a_t) S_N + ks_t^T v_t                       (shared)
    o_t  = sum_{i in T_t} e_t[i] scale q_t S_i + scale qs_t S_N

for the loss L = sum(d_out * o) + sum(d_final_state * S_final).  The notes
(section 2.3) point out that the same e_t[i] appears at the write and at the
read, so the router weight receives gradient from both; the top-k indices
are piecewise constant and carry none, and the softmax is over all N
partitions, so d l_t = e_t * (de_t - <e_t, de_t>) with de_t[i] = 0 for the
unselected i.

Reverse pass (per sequence and head, t from last to first), with
G_i = dL/dS_i after step t:
    read :  G_i += e_i scale q_t^T do_t;   dq_t += e_i scale S_i do_t^T;
            de_i += scale q_t S_i do_t^T                     (S_i after step t)
    write:  dk_t += e_i G_i v_t^T;   dv_t += e_i k_t G_i;   de_i += k_t G_i v_t^T;
            da_t += rowsum(G_i * S_i before step t);   G_i <- diag(a_t) G_i
and the same for the shared slot with weight 1 (qs, ks); dg_t = a_t * da_t;
d initial_state = G after the first token.

Parity status: pinned by ``tests/test_oracle_backward.py`` against central
finite differences of the forward oracle (the C recurrence), the shift
invariance of the router softmax, and planted-mistake checks.
"""
from __future__ import annotations

import numpy as np

from . import to_f64


def _softmax(x):
    z = np.exp(x - x.max())
    return z / z.sum()


def _topk(l, k):
    return np.argsort(-l, kind="stable")[:k]


def backward(q, k, v, g, logits, cu_seqlens, d_out, *, top_k: int, use_shared: int = 1, scale: float = 1.0,
             q_shared=None, k_shared=None, initial_state=None, d_final_state=None) -> dict:
    """Gradients of L = sum(d_out * out) + sum(d_final_state * final_state).
    Arrays [T, H, .] (states [S, H, P, c, d]); returns dq, dk, dv, dg,
    dlogits, dq_shared / dk_shared (None when the shared q / k are q / k, whose
    gradients then include the shared terms), d_initial_state, and the
    recomputed out / final_state."""
    Q, K, V, Gt, Lg, dO = (to_f64(x) for x in (q, k, v, g, logits, d_out))
    QS = Q if q_shared is None else to_f64(q_shared)
    KS = K if k_shared is None else to_f64(k_shared)
    T, H, c = Q.shape
    d = V.shape[2]
    N = Lg.shape[2]
    P = N + (1 if use_shared else 0)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    S_n = len(cu) - 1
    init = None if initial_state is None else to_f64(initial_state)
    dfin = None if d_final_state is None else to_f64(d_final_state)

    dq, dk, dv, dg, dl = (np.zeros_like(x) for x in (Q, K, V, Gt, Lg))
    dqs, dks = np.zeros_like(QS), np.zeros_like(KS)
    dinit = np.zeros((S_n, H, P, c, d))
    out = np.zeros((T, H, d))
    fin = np.zeros((S_n, H, P, c, d))

    for b in range(S_n):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        for h in range(H):
            S = np.zeros((P, c, d)) if init is None else init[b, h].copy()
            rec = []
            for t in range(t0, t1):
                e = _softmax(Lg[t, h])
                sel = _topk(Lg[t, h], top_k)
                a = np.exp(Gt[t, h])
                before = S.copy()
                for i in sel:
                    S[i] = a[:, None] * S[i] + e[i] * np.outer(K[t, h], V[t, h])
                if use_shared:
                    S[N] = a[:, None] * S[N] + np.outer(KS[t, h], V[t, h])
                o = sum(e[i] * scale * (Q[t, h] @ S[i]) for i in sel)
                if use_shared:
                    o = o + scale * (QS[t, h] @ S[N])
                out[t, h] = o
                rec.append((before, S.copy(), e, sel, a))
            fin[b, h] = S
            G = np.zeros((P, c, d)) if dfin is None else dfin[b, h].copy()
            for t in range(t1 - 1, t0 - 1, -1):
                before, after, e, sel, a = rec[t - t0]
                do = dO[t, h]
                de = np.zeros(N)
                # read at step t (post-update states)
                for i in sel:
                    G[i] += e[i] * scale * np.outer(Q[t, h], do)
                    dq[t, h] += e[i] * scale * (after[i] @ do)
                    de[i] += scale * (Q[t, h] @ after[i] @ do)
                if use_shared:
                    G[N] += scale * np.outer(QS[t, h], do)
                    dqs[t, h] += scale * (after[N] @ do)
                # write and decay at step t
                da = np.zeros(c)
                for i in sel:
                    dk[t, h] += e[i] * (G[i] @ V[t, h])
                    dv[t, h] += e[i] * (K[t, h] @ G[i])
                    de[i] += K[t, h] @ G[i] @ V[t, h]
                    da += (G[i] * before[i]).sum(axis=1)
                    G[i] = a[:, None] * G[i]
                if use_shared:
                    dks[t, h] += G[N] @ V[t, h]
                    dv[t, h] += KS[t, h] @ G[N]
                    da += (G[N] * before[N]).sum(axis=1)
                    G[N] = a[:, None] * G[N]
                dg[t, h] = da * a
                dl[t, h] = e * (de - e @ de)
            dinit[b, h] = G

    res = {"dq": dq, "dk": dk, "dv": dv, "dg": dg, "dlogits": dl, "d_initial_state": dinit,
           "out": out, "final_state": fin, "dq_shared": None, "dk_shared": None}
    if q_shared is None:
        res["dq"] = dq + dqs
    else:
        res["dq_shared"] = dqs
    if k_shared is None:
        res["dk"] = dk + dks
    else:
        res["dk_shared"] = dks
    return res
