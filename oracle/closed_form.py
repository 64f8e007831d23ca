"""Brute-force unrolled forms of the SSE layer -- TEST INFRASTRUCTURE.

``closed_form`` writes the layer output as the double sum of "Scaling Linear
Attention with Sparse State Expansion" (close-reading notes, section 2.4, the
unrolled form of eqs. 13-14): a past token s reaches the output of token t
only through partitions selected at both t and s, weighted by the router
probability at both ends, and decayed only by the gates of the steps in
(s, t] at which that partition was selected.  It adds the always-on shared
partition (section 2.5; decayed at every step, weight 1) and the contribution
of an initial state, which the page's derivation omits by starting from zero.

Routing here is computed independently of the C oracle: a numpy softmax and
a stable argsort of the negated logits (equal logits keep ascending index).

``dense_gla`` is gated linear attention in its quadratic masked form,
o_t = sum_{s<=t} sum_r q_t[r] k_s[r] exp(G_t[r] - G_s[r]) v_s with G the
running sum of the log gates (section 2.1, eq. 6 with a diagonal transition).
"""
from __future__ import annotations

import numpy as np


def _route(logits_th: np.ndarray, top_k: int):
    """logits [T, N] -> (e [T, N] softmax, sel [T, N] bool of the top-k)."""
    z = logits_th - logits_th.max(axis=1, keepdims=True)
    ez = np.exp(z)
    e = ez / ez.sum(axis=1, keepdims=True)
    order = np.argsort(-logits_th, axis=1, kind="stable")[:, :top_k]
    sel = np.zeros_like(logits_th, dtype=bool)
    np.put_along_axis(sel, order, True, axis=1)
    return e, sel


def closed_form(q, k, v, g, logits, cu_seqlens, *, top_k, use_shared=1, scale=1.0,
                q_shared=None, k_shared=None, initial_state=None):
    """float64 arrays [T, H, .] -> out [T, H, d].  Intended for T <= ~64."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    logits = np.asarray(logits, np.float64)
    qs = q if q_shared is None else np.asarray(q_shared, np.float64)
    ks = k if k_shared is None else np.asarray(k_shared, np.float64)
    T, H, c = q.shape
    d = v.shape[2]
    N = logits.shape[2]
    out = np.zeros((T, H, d))
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    for b in range(len(cu) - 1):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        L = t1 - t0
        if L == 0:
            continue
        causal = np.tril(np.ones((L, L), dtype=bool))
        for h in range(H):
            qb, kb, vb, gb = q[t0:t1, h], k[t0:t1, h], v[t0:t1, h], g[t0:t1, h]
            e, sel = _route(logits[t0:t1, h], top_k)
            o = np.zeros((L, d))
            for i in range(N):
                # log-decay accumulated only over the steps that selected i
                Li = np.cumsum(gb * sel[:, i:i + 1], axis=0)            # [L, c]
                dec = np.exp(Li[:, None, :] - Li[None, :, :])           # [t, s, c]
                A = np.einsum("tr,sr,tsr->ts", qb, kb, dec)
                w = (sel[:, i] * e[:, i])[:, None] * (sel[:, i] * e[:, i])[None, :]
                o += (A * w * causal) @ vb
                if initial_state is not None:
                    S0 = np.asarray(initial_state[b, h, i], np.float64)
                    o += (sel[:, i] * e[:, i])[:, None] * ((qb * np.exp(Li)) @ S0)
            if use_shared:
                qsb, ksb = qs[t0:t1, h], ks[t0:t1, h]
                Ls = np.cumsum(gb, axis=0)
                dec = np.exp(Ls[:, None, :] - Ls[None, :, :])
                A = np.einsum("tr,sr,tsr->ts", qsb, ksb, dec)
                o += (A * causal) @ vb
                if initial_state is not None:
                    S0 = np.asarray(initial_state[b, h, N], np.float64)
                    o += (qsb * np.exp(Ls)) @ S0
            out[t0:t1, h] = scale * o
    return out


def dense_gla(q, k, v, g, cu_seqlens):
    """Quadratic masked gated linear attention, float64, arrays [T, H, .]."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    T, H, c = q.shape
    out = np.zeros((T, H, v.shape[2]))
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    for b in range(len(cu) - 1):
        t0, t1 = int(cu[b]), int(cu[b + 1])
        L = t1 - t0
        if L == 0:
            continue
        causal = np.tril(np.ones((L, L)))
        for h in range(H):
            G = np.cumsum(g[t0:t1, h], axis=0)
            dec = np.exp(G[:, None, :] - G[None, :, :])
            A = np.einsum("tr,sr,tsr->ts", q[t0:t1, h], k[t0:t1, h], dec)
            out[t0:t1, h] = (A * causal) @ v[t0:t1, h]
    return out
