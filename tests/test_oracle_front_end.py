"""Pins of the front-end oracle (CPU only): eqs. 9-10 of "Scaling Linear
Attention with Sparse State Expansion" (close-reading notes, section 2.3),
GLA's log-gate, and the shared partition's rank-64 Q/K LoRA (section 2.5).

Each pin checks the oracle against a value fixed by the mathematics, not by
the oracle's own formula: identity and permutation weights (orientation of
y = x W^T), uniform keys from zero key weights, closed forms of the softmax and
logsigmoid, and LoRA cases whose result is known in closed form.  The mutation
cases at the end plant one plausible mistake at a time and check that some pin
sees it.
"""
import math

import numpy as np
import pytest

from oracle import front_end as fe

RNG = np.random.default_rng(7)


def _weights(H, c, d, N, D, rng=RNG):
    return dict(w_q=rng.normal(size=(H * c, D)), w_k=rng.normal(size=(H * c, D)),
                w_v=rng.normal(size=(H * d, D)), w_g=rng.normal(size=(H * c, D)),
                w_e=rng.normal(size=(H * N, D)))


def test_identity_and_permutation_weights(fn=None):
    """W_q = I gives q = x; W_v = a row permutation P gives v[:, n] = x[:, perm[n]]
    (a transposed product would give the inverse permutation); one-hot router
    rows pick single features of x."""
    fn = fn or fe.front_end
    H, c, N = 2, 3, 2
    D = H * c
    T = 4
    x = RNG.normal(size=(T, D))
    perm = np.array([1, 2, 3, 4, 5, 0])          # a 6-cycle: not its own inverse
    w = _weights(H, c, c, N, D)
    w["w_q"] = np.eye(D)
    w["w_v"] = np.eye(D)[perm]
    w["w_e"] = np.zeros((H * N, D))
    w["w_e"][np.arange(H * N), [5, 0, 2, 4]] = 1.0
    out = fn(x, **w, num_heads=H)
    assert np.array_equal(out["q"].reshape(T, D), x)
    assert np.array_equal(out["v"].reshape(T, D), x[:, perm])
    assert np.array_equal(out["logits"].reshape(T, H * N), x[:, [5, 0, 2, 4]])


def test_key_softmax_closed_forms(fn=None):
    """Zero key weights give uniform keys 1/c; a single active key logit a
    gives e^a / (e^a + c - 1) there and 1 / (e^a + c - 1) elsewhere."""
    fn = fn or fe.front_end
    H, c, N, D, T = 2, 4, 2, 5, 3
    x = RNG.normal(size=(T, D))
    w = _weights(H, c, c, N, D)
    w["w_k"] = np.zeros((H * c, D))
    out = fn(x, **w, num_heads=H)
    assert np.allclose(out["k"], 1.0 / c, rtol=0, atol=1e-15)
    w["w_k"][2, 0] = 1.0                          # head 0, key row 2 <- x[:, 0]
    out = fn(x, **w, num_heads=H)
    a = x[:, 0]
    den = np.exp(a) + c - 1
    assert np.allclose(out["k"][:, 0, 2], np.exp(a) / den, rtol=1e-14)
    assert np.allclose(out["k"][:, 0, 0], 1.0 / den, rtol=1e-14)
    assert np.allclose(out["k"][:, 1, :], 1.0 / c, rtol=0, atol=1e-15)


def test_gate_closed_forms(fn=None):
    """g = logsigmoid(y) / tau: exactly -ln 2 / tau at y = 0; the identity
    logsigmoid(y) - logsigmoid(-y) = y; the limits -e^{-y} (y -> +inf) and
    y - e^{y} (y -> -inf)."""
    fn = fn or fe.front_end
    H, c, N, D, T = 1, 4, 2, 4, 5
    x = np.array([[0.0, 0.0, 0.0, 0.0], [1.0, -2.0, 30.0, -30.0],
                  [0.5, 3.0, -0.25, 7.0], [-1.0, 1.0, 2.0, -2.0], [4.0, -4.0, 0.0, 0.0]])
    w = _weights(H, c, c, N, D)
    w["w_g"] = np.eye(D)
    out = fn(x, **w, num_heads=H, gate_inv_tau=1.0 / 16)
    g = out["g"][:, 0, :] * 16
    assert np.all(g[0] == -math.log(2.0))
    assert abs(g[1, 2] + math.exp(-30.0)) < 1e-25
    assert abs(g[1, 3] - (-30.0 - math.exp(-30.0))) < 1e-12
    w["w_g"] = -np.eye(D)
    gm = fn(x, **w, num_heads=H, gate_inv_tau=1.0 / 16)["g"][:, 0, :] * 16
    assert np.allclose(g - gm, x, rtol=0, atol=1e-13)
    assert np.all(g <= 0)


def test_lora_special_cases(fn=None):
    """B = 0: the shared q/k equal the routed ones.  D = r, A = I, B = W: the
    shared query is 2q and the shared key softmax(2 y_k) = k^2 / sum(k^2)."""
    fn = fn or fe.front_end
    H, c, N, T = 2, 3, 2, 4
    r = D = 6
    x = RNG.normal(size=(T, D))
    w = _weights(H, c, c, N, D)
    zero = dict(a_q=RNG.normal(size=(r, D)), b_q=np.zeros((H * c, r)),
                a_k=RNG.normal(size=(r, D)), b_k=np.zeros((H * c, r)))
    out = fn(x, **w, num_heads=H, **zero)
    assert np.array_equal(out["q_shared"], out["q"])
    assert np.allclose(out["k_shared"], out["k"], rtol=1e-15, atol=0)
    dbl = dict(a_q=np.eye(D), b_q=w["w_q"], a_k=np.eye(D), b_k=w["w_k"])
    out = fn(x, **w, num_heads=H, **dbl)
    assert np.allclose(out["q_shared"], 2 * out["q"], rtol=1e-14)
    k2 = out["k"] ** 2
    assert np.allclose(out["k_shared"], k2 / k2.sum(-1, keepdims=True), rtol=1e-12)
    none = fn(x, **w, num_heads=H)
    assert none["q_shared"] is None and none["k_shared"] is None


PINS = [test_identity_and_permutation_weights, test_key_softmax_closed_forms, test_gate_closed_forms,
        test_lora_special_cases]


def _mutant(kind):
    """A copy of the oracle with one planted mistake."""
    def fn(x, w_q, w_k, w_v, w_g, w_e, *, num_heads, gate_inv_tau=1.0 / 16, a_q=None, b_q=None, a_k=None,
           b_k=None):
        if kind == "transposed_value_weights":
            w_v = np.asarray(w_v).T
        if kind == "gate_without_tau":
            gate_inv_tau = 1.0
        if kind == "lora_on_value_side":
            b_q = None if b_q is None else np.asarray(b_q) * 0.0
        out = fe.front_end(x, w_q, w_k, w_v, w_g, w_e, num_heads=num_heads, gate_inv_tau=gate_inv_tau,
                           a_q=a_q, b_q=b_q, a_k=a_k, b_k=b_k)
        T, H = out["q"].shape[:2]
        if kind == "key_softmax_over_heads":
            y = np.log(out["k"])
            out["k"] = fe.softmax_last(np.swapaxes(y, 1, 2)).swapaxes(1, 2)
        if kind == "gate_sigmoid_not_log":
            out["g"] = np.exp(out["g"] / gate_inv_tau) * gate_inv_tau
        if kind == "shared_key_not_renormalised" and out["k_shared"] is not None:
            out["k_shared"] = out["k_shared"] * 1.5
        return out
    return fn


@pytest.mark.parametrize("kind", ["transposed_value_weights", "gate_without_tau", "lora_on_value_side",
                                  "key_softmax_over_heads", "gate_sigmoid_not_log",
                                  "shared_key_not_renormalised"])
def test_front_end_mutant_is_killed(kind):
    fn = _mutant(kind)
    failed = 0
    for pin in PINS:
        try:
            pin(fn)
        except (AssertionError, ValueError):
            failed += 1
    assert failed > 0, f"mutant {kind} survived every pin"
