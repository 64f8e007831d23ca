"""Pins of the delta-rule SSE oracle (``oracle/delta.py``), CPU only.

Each pin checks the oracle against something other than itself:
- beta = 0: no write at all, each selected step multiplies the state by its
  alpha -- a closed form of the initial state;
- exact retrieval (DeltaNet, "动态线性注意力" section 2.1, eq. 4): with a unit
  key, beta = 1, alpha = 1 and one partition, the state answers the key just
  written with its value, q = k -> o = v, whatever it held before;
- the product form: one partition, no shared one, S_T = A_T ... A_1 S_0 + sum_t
  (A_T ... A_{t+1}) beta_t k_t^T v_t with A_t = alpha_t (I - beta_t k_t^T k_t),
  written as numpy matrix products;
- top_k = N with equal logits: every partition holds the same state, the
  routed read-out is the single-partition delta rule with beta / N;
- partitions never selected keep their initial state bit for bit;
- planted mistakes in a copy of the oracle's source each fail a pin.
"""
import inspect
import types

import numpy as np

from oracle import delta as dl


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _case(rng, T, H, c, d, N, *, beta=None, alpha=None):
    q = rng.normal(size=(T, H, c)) / np.sqrt(c)
    k = _unit(rng.normal(size=(T, H, c)))
    v = rng.normal(size=(T, H, d))
    la = np.log(alpha) * np.ones((T, H)) if alpha is not None else -np.abs(rng.normal(size=(T, H))) * 0.2
    b = beta * np.ones((T, H)) if beta is not None else 1.0 / (1.0 + np.exp(-rng.normal(size=(T, H))))
    logits = rng.normal(size=(T, H, N))
    return q, k, v, la, b, logits


def test_beta_zero_is_decay_only(mod=dl):
    rng = np.random.default_rng(0)
    T, H, c, d, N, K = 9, 2, 4, 3, 4, 2
    q, k, v, la, b, logits = _case(rng, T, H, c, d, N, beta=0.0)
    init = rng.normal(size=(1, H, N + 1, c, d))
    cu = np.array([0, T])
    r = mod.delta_forward(q, k, v, la, b, logits, cu, top_k=K, use_shared=1, initial_state=init)
    for h in range(H):
        fac = np.ones(N + 1)
        for t in range(T):
            sel = np.argsort(-logits[t, h], kind="stable")[:K]
            fac[sel] *= np.exp(la[t, h])
            fac[N] *= np.exp(la[t, h])
            e = np.exp(logits[t, h] - logits[t, h].max())
            e /= e.sum()
            o = sum(e[i] * q[t, h] @ (fac[i] * init[0, h, i]) for i in sel) + q[t, h] @ (fac[N] * init[0, h, N])
            np.testing.assert_allclose(r["out"][t, h], o, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["final_state"][0, h], fac[:, None, None] * init[0, h], rtol=1e-12, atol=1e-14)


def test_exact_retrieval_of_the_last_write(mod=dl):
    rng = np.random.default_rng(1)
    T, H, c, d = 12, 1, 6, 5
    _, k, v, la, b, logits = _case(rng, T, H, c, d, 1, beta=1.0, alpha=1.0)
    init = rng.normal(size=(1, H, 1, c, d))
    r = mod.delta_forward(k.copy(), k, v, la, b, logits, np.array([0, T]), top_k=1, use_shared=0,
                          initial_state=init)
    # e = 1 (one partition): o_t = k_t S_t = v_t exactly
    np.testing.assert_allclose(r["out"], v, rtol=1e-12, atol=1e-12)


def _product_form(k, v, la, b, S0):
    S = S0.copy()
    c = S.shape[0]
    for t in range(k.shape[0]):
        A = np.exp(la[t]) * (np.eye(c) - b[t] * np.outer(k[t], k[t]))
        S = A @ S + b[t] * np.outer(k[t], v[t])
    return S


def test_product_form_single_partition(mod=dl):
    rng = np.random.default_rng(2)
    T, H, c, d = 15, 2, 5, 4
    q, k, v, la, b, logits = _case(rng, T, H, c, d, 1)
    init = rng.normal(size=(2, H, 1, c, d))
    cu = np.array([0, 6, T])
    r = mod.delta_forward(q, k, v, la, b, logits, cu, top_k=1, use_shared=0, scale=0.7, initial_state=init)
    for s in range(2):
        t0, t1 = cu[s], cu[s + 1]
        for h in range(H):
            S_end = _product_form(k[t0:t1, h], v[t0:t1, h], la[t0:t1, h], b[t0:t1, h], init[s, h, 0])
            np.testing.assert_allclose(r["final_state"][s, h, 0], S_end, rtol=1e-11, atol=1e-12)
            # read after write at every step: o_t = 0.7 q_t S_t
            for t in range(t0, t1):
                St = _product_form(k[t0:t + 1, h], v[t0:t + 1, h], la[t0:t + 1, h], b[t0:t + 1, h], init[s, h, 0])
                np.testing.assert_allclose(r["out"][t, h], 0.7 * q[t, h] @ St, rtol=1e-11, atol=1e-12)


def test_k_equals_n_equal_logits(mod=dl):
    rng = np.random.default_rng(3)
    T, H, c, d, N = 10, 1, 4, 4, 4
    q, k, v, la, b, _ = _case(rng, T, H, c, d, N)
    logits = np.zeros((T, H, N))
    r = mod.delta_forward(q, k, v, la, b, logits, np.array([0, T]), top_k=N, use_shared=0)
    # every partition: the delta rule with beta / N; routed read-out = q S (N terms of 1/N)
    for t in range(T):
        St = _product_form(k[:t + 1, 0], v[:t + 1, 0], la[:t + 1, 0], b[:t + 1, 0] / N, np.zeros((c, d)))
        np.testing.assert_allclose(r["out"][t, 0], q[t, 0] @ St, rtol=1e-11, atol=1e-12)
    for i in range(N):
        np.testing.assert_allclose(r["final_state"][0, 0, i], St, rtol=1e-11, atol=1e-12)


def test_unselected_partitions_untouched(mod=dl):
    rng = np.random.default_rng(4)
    T, H, c, d, N = 8, 2, 4, 3, 6
    q, k, v, la, b, logits = _case(rng, T, H, c, d, N)
    logits[..., 4:] = -50.0
    init = rng.normal(size=(1, H, N + 1, c, d))
    r = mod.delta_forward(q, k, v, la, b, logits, np.array([0, T]), top_k=2, use_shared=1, initial_state=init)
    assert np.array_equal(r["final_state"][0, :, 4:6], init[0, :, 4:6])
    # decode: one step on the same states leaves them untouched too
    st = r["final_state"].copy()
    dl.delta_decode_step(st, q[:1], k[:1], v[:1], la[:1], b[:1], logits[:1], top_k=2)
    assert np.array_equal(st[0, :, 4:6], init[0, :, 4:6])


def test_decode_continues_the_forward():
    rng = np.random.default_rng(5)
    T, H, c, d, N = 11, 2, 4, 3, 5
    q, k, v, la, b, logits = _case(rng, T, H, c, d, N)
    full = dl.delta_forward(q, k, v, la, b, logits, np.array([0, T]), top_k=2)
    head = dl.delta_forward(q[:8], k[:8], v[:8], la[:8], b[:8], logits[:8], np.array([0, 8]), top_k=2)
    st = head["final_state"].copy()
    for t in range(8, T):
        o = dl.delta_decode_step(st, q[t:t + 1], k[t:t + 1], v[t:t + 1], la[t:t + 1], b[t:t + 1], logits[t:t + 1],
                                 top_k=2)
        np.testing.assert_allclose(o["out"][0], full["out"][t], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(st, full["final_state"], rtol=1e-12, atol=1e-12)


MUTANTS = {
    "erase_without_router_weight": ("S[i] - e * b * np.outer(k, k @ S[i])", "S[i] - b * np.outer(k, k @ S[i])"),
    "write_not_decayed_erase": ("a * (S[i] - e * b * np.outer(k, k @ S[i]))", "a * S[i] - e * b * np.outer(k, k @ S[i])"),
    "write_without_beta": ("+ e * b * np.outer(k, v)", "+ e * np.outer(k, v)"),
    "erase_missing": ("S[i] - e * b * np.outer(k, k @ S[i])", "S[i]"),
    "alpha_inverted": ("np.exp(LA[t, h])", "np.exp(-LA[t, h])"),
}
# a copy with a no-op edit: the harness itself leaves a correct oracle passing
CONTROL = ("o = sum(e * scale * (q @ S[i]) for i, e in zip(sel, e_sel))\n",
           "o = sum(e * scale * (q @ S[i]) for i, e in zip(sel, e_sel)) * 1.0\n")


def _mutant(old, new):
    src = inspect.getsource(dl)
    assert old in src, old
    mod = types.ModuleType("delta_mutant")
    mod.__dict__["to_f64"] = dl.to_f64
    exec(compile(src.replace(old, new, 1).replace("from . import to_f64", ""), "delta_mutant", "exec"), mod.__dict__)
    return mod


def test_planted_mistakes_are_caught():
    pins = (test_beta_zero_is_decay_only, test_exact_retrieval_of_the_last_write, test_product_form_single_partition,
            test_k_equals_n_equal_logits, test_unselected_partitions_untouched)
    survived = []
    for name, (old, new) in MUTANTS.items():
        mod = _mutant(old, new)
        caught = False
        for pin in pins:
            try:
                pin(mod)
            except AssertionError:
                caught = True
                break
        if not caught:
            survived.append(name)
    assert not survived, survived
    mod = _mutant(*CONTROL)
    for pin in pins:
        pin(mod)
