"""Pins of the backward oracle (CPU only).

The gradients of the backward oracle (``oracle/backward.py``) are checked
against central finite differences of the forward oracle (the C recurrence of
``oracle/sse_oracle.c``, a separate implementation), for every input: q, k, v,
the log-gate, the router logits, separate shared q / k, and the initial state,
with a loss that weighs both the outputs and the final states.  Logits are
well separated so that no perturbation changes a top-k selection.  Further
pins: the router softmax is invariant to adding a constant to a token's logits,
so each token's logit gradient sums to zero; the recomputed forward equals the
C forward.  The mutation cases plant one plausible mistake at a time in a copy
of the backward's source and check that a pin sees it.
"""
import inspect

import numpy as np
import pytest

import oracle
from oracle import backward as bw

H, c, d, N, K = 2, 3, 2, 4, 2
CU = np.array([0, 4, 7], dtype=np.int64)
T, S = int(CU[-1]), len(CU) - 1


def _case(seed=0, use_shared=1, separate_shared=True):
    rng = np.random.default_rng(seed)
    P = N + use_shared
    x = dict(
        q=rng.normal(size=(T, H, c)), k=rng.normal(size=(T, H, c)) * 0.5, v=rng.normal(size=(T, H, d)),
        g=-np.abs(rng.normal(size=(T, H, c))) * 0.3,
        # a random order of 0..N-1 per token: top-k margins of about 1 >> the step
        logits=np.stack([np.stack([rng.permutation(N) + rng.normal(scale=0.01, size=N) for _ in range(H)])
                         for _ in range(T)]).astype(np.float64),
        q_shared=rng.normal(size=(T, H, c)) if (use_shared and separate_shared) else None,
        k_shared=rng.normal(size=(T, H, c)) * 0.5 if (use_shared and separate_shared) else None,
        initial_state=rng.normal(size=(S, H, P, c, d)) * 0.3,
    )
    d_out = rng.normal(size=(T, H, d))
    d_fin = rng.normal(size=(S, H, P, c, d))
    return x, d_out, d_fin


def _loss(x, d_out, d_fin, use_shared, scale):
    f = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["logits"], CU, top_k=K, use_shared=use_shared,
                       scale=scale, q_shared=x["q_shared"], k_shared=x["k_shared"],
                       initial_state=x["initial_state"])
    return float(np.sum(d_out * f["out"]) + np.sum(d_fin * f["final_state"]))


def _grads(fn, x, d_out, d_fin, use_shared, scale):
    return fn(x["q"], x["k"], x["v"], x["g"], x["logits"], CU, d_out, top_k=K, use_shared=use_shared, scale=scale,
              q_shared=x["q_shared"], k_shared=x["k_shared"], initial_state=x["initial_state"],
              d_final_state=d_fin)


GRAD_OF = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "logits": "dlogits", "q_shared": "dq_shared",
           "k_shared": "dk_shared", "initial_state": "d_initial_state"}


@pytest.mark.parametrize("use_shared,separate,scale", [(1, True, 1.0), (1, False, 0.7), (0, False, 1.0)])
def test_backward_matches_finite_differences(use_shared, separate, scale, fn=None):
    """Every gradient equals the central difference of the forward oracle's
    loss (step 1e-6, float64) to 1e-6 relative."""
    fn = fn or bw.backward
    x, d_out, d_fin = _case(1, use_shared, separate)
    got = _grads(fn, x, d_out, d_fin, use_shared, scale)
    eps = 1e-6
    for name, gname in GRAD_OF.items():
        if x[name] is None:
            assert got[gname] is None or gname in ("dq_shared", "dk_shared")
            continue
        base = x[name]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            old = base[idx]
            base[idx] = old + eps
            lp = _loss(x, d_out, d_fin, use_shared, scale)
            base[idx] = old - eps
            lm = _loss(x, d_out, d_fin, use_shared, scale)
            base[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        g = got[gname]
        err = np.max(np.abs(g - fd)) / max(np.max(np.abs(fd)), 1e-12)
        assert err < 1e-6, (name, err)


def test_logit_gradient_sums_to_zero(fn=None):
    """softmax(l + const) = softmax(l): each token's logit gradient sums to 0."""
    fn = fn or bw.backward
    x, d_out, d_fin = _case(2)
    got = _grads(fn, x, d_out, d_fin, 1, 1.0)
    assert np.max(np.abs(got["dlogits"].sum(axis=-1))) < 1e-12
    assert np.max(np.abs(got["dlogits"])) > 1e-3


def test_recomputed_forward_matches_c_oracle():
    x, d_out, d_fin = _case(3)
    got = _grads(bw.backward, x, d_out, d_fin, 1, 1.0)
    f = oracle.forward(x["q"], x["k"], x["v"], x["g"], x["logits"], CU, top_k=K, use_shared=1,
                       q_shared=x["q_shared"], k_shared=x["k_shared"], initial_state=x["initial_state"])
    assert np.allclose(got["out"], f["out"], rtol=1e-12, atol=1e-12)
    assert np.allclose(got["final_state"], f["final_state"], rtol=1e-12, atol=1e-12)


MUTANTS = {
    "no_decay_of_state_gradient": ("G[i] = a[:, None] * G[i]", "G[i] = G[i]"),
    "read_uses_state_before_update": ("dq[t, h] += e[i] * scale * (after[i] @ do)",
                                      "dq[t, h] += e[i] * scale * (before[i] @ do)"),
    "router_weight_only_at_read": ("de[i] += K[t, h] @ G[i] @ V[t, h]", "de[i] += 0.0"),
    "softmax_jacobian_not_centred": ("dl[t, h] = e * (de - e @ de)", "dl[t, h] = e * de"),
    "gate_gradient_missing_a": ("dg[t, h] = da * a", "dg[t, h] = da"),
    "shared_key_gradient_unweighted_value": ("dks[t, h] += G[N] @ V[t, h]", "dks[t, h] += G[N].sum(axis=1)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_backward_mutant_is_killed(name):
    old, new = MUTANTS[name]
    src = inspect.getsource(bw)
    assert src.count(old) == 1, name
    ns = {"__name__": "oracle.backward_mutant"}
    src = src.replace("from . import to_f64", "from oracle import to_f64").replace(old, new)
    exec(compile(src, "backward_mutant", "exec"), ns)
    fn = ns["backward"]
    killed = False
    for pin in (lambda: test_backward_matches_finite_differences(1, True, 1.0, fn=fn),
                lambda: test_logit_gradient_sums_to_zero(fn=fn)):
        try:
            pin()
        except AssertionError:
            killed = True
    assert killed, f"mutant {name} survived every pin"
