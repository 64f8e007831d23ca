"""Front end of the SSE layer -- TEST INFRASTRUCTURE (float64, numpy).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU leg may
use this module; the CUDA library shares no code with it.

"Scaling Linear Attention with Sparse State Expansion" (close-reading notes,
section 2.3, eqs. 9-10) gives the per-token projections feeding the state
update, per head:

    e_t = softmax(x_t W_e)            (the router; the layer takes the logits)
    q_t = x_t W_q,   v_t = x_t W_v,   k_t = softmax(x_t W_k)   (over the c keys)

and section 2.5 gives the always-on shared partition its own Q/K through a
rank-64 LoRA of the same projections (V stays shared):

    q^s_t = x_t W_q + (x_t A_q) B_q,     k^s_t = softmax(x_t W_k + (x_t A_k) B_k).

The diagonal gate is GLA's (notes section 2.1): a decay
alpha = sigmoid(x_t W_g)^(1/tau), i.e. the log-gate g = logsigmoid(x_t W_g) / tau
(tau = 16 in GLA and in the synthetic workloads' gate recipe).

Weights use the [out_features, in_features] layout (y = x W^T):
w_q, w_k, w_g [H*c, D]; w_v [H*d, D]; w_e [H*N, D]; a_q, a_k [r, D];
b_q, b_k [H*c, r].  Every matrix product here is a plain float64 matmul.

Parity status: pinned by ``tests/test_oracle_front_end.py`` (identity and
permutation weights, uniform keys and the exact gate at zero, LoRA special
cases, the sigmoid/logsigmoid limits).
"""
from __future__ import annotations

import numpy as np

from . import to_f64


def logsigmoid(y: np.ndarray) -> np.ndarray:
    """log(1 / (1 + exp(-y))), evaluated without overflow for either sign."""
    y = np.asarray(y, dtype=np.float64)
    return np.where(y >= 0, -np.log1p(np.exp(-np.abs(y))), y - np.log1p(np.exp(-np.abs(y))))


def softmax_last(y: np.ndarray) -> np.ndarray:
    """Softmax over the last axis (max subtracted first)."""
    m = y.max(axis=-1, keepdims=True)
    z = np.exp(y - m)
    return z / z.sum(axis=-1, keepdims=True)


def front_end(x, w_q, w_k, w_v, w_g, w_e, *, num_heads: int, gate_inv_tau: float = 1.0 / 16.0,
              a_q=None, b_q=None, a_k=None, b_k=None) -> dict:
    """x [T, D] -> q, k, g [T, H, c]; v [T, H, d]; logits [T, H, N]; and, when
    the LoRA factors are given, q_shared / k_shared [T, H, c] (else None).
    Inputs may be bfloat16 bit patterns (uint16) or floats."""
    H = num_heads
    X = to_f64(x)
    T = X.shape[0]

    def proj(w):
        return X @ to_f64(w).T

    yq, yk, yv, yg, ye = proj(w_q), proj(w_k), proj(w_v), proj(w_g), proj(w_e)
    c = yq.shape[1] // H
    out = {
        "q": yq.reshape(T, H, c),
        "k": softmax_last(yk.reshape(T, H, c)),
        "v": yv.reshape(T, H, -1),
        "g": logsigmoid(yg.reshape(T, H, c)) * gate_inv_tau,
        "logits": ye.reshape(T, H, -1),
        "q_shared": None,
        "k_shared": None,
    }
    if a_q is not None:
        lq = (X @ to_f64(a_q).T) @ to_f64(b_q).T
        lk = (X @ to_f64(a_k).T) @ to_f64(b_k).T
        out["q_shared"] = (yq + lq).reshape(T, H, c)
        out["k_shared"] = softmax_last((yk + lk).reshape(T, H, c))
    return out
