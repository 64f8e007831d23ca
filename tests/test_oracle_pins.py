"""Pins of the fp64 CPU oracle against facts fixed by the source pages and by
mathematics, independent of the oracle's own code (CPU only).

Source: "Scaling Linear Attention with Sparse State Expansion" (close-reading
notes), sections 1-2.6; plain linear attention also from "Dynamic Linear
Attention" section 2.1, eqs. 1-3.
"""
import json
import os

import numpy as np
import pytest

import oracle
from sparse_state_linear_router_gb300 import inputs as synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(rng, lengths, H, c, d, N, with_init=True, shared_qk=True):
    T = int(sum(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    q = rng.normal(size=(T, H, c))
    k = rng.random(size=(T, H, c)) + 0.05
    v = rng.normal(size=(T, H, d))
    g = -rng.random(size=(T, H, c)) * 0.5
    logits = rng.normal(size=(T, H, N))
    P = N + 1
    init = rng.normal(size=(len(lengths), H, P, c, d)) * 0.3 if with_init else None
    qs = None if shared_qk else rng.normal(size=(T, H, c))
    ks = None if shared_qk else rng.random(size=(T, H, c))
    return dict(q=q, k=k, v=v, g=g, logits=logits, cu=cu, init=init, qs=qs, ks=ks)


def test_textbook_linear_attention():
    """N=1, k=1, no shared partition, zero log-gate: the layer is plain causal
    linear attention o = (Q K^T * causal mask) V (pages: SSE notes section 1;
    Dynamic Linear Attention eq. 1).  Keys here are arbitrary, not softmaxed."""
    rng = np.random.default_rng(1)
    lengths = [7, 0, 13, 1]
    T, H, c, d = sum(lengths), 2, 5, 3
    cu = np.concatenate([[0], np.cumsum(lengths)])
    q, k, v = rng.normal(size=(T, H, c)), rng.normal(size=(T, H, c)), rng.normal(size=(T, H, d))
    g = np.zeros((T, H, c))
    logits = rng.normal(size=(T, H, 1))
    res = oracle.forward(q, k, v, g, logits, cu, top_k=1, use_shared=0)
    for b in range(len(lengths)):
        t0, t1 = cu[b], cu[b + 1]
        for h in range(H):
            Q, K, V = q[t0:t1, h], k[t0:t1, h], v[t0:t1, h]
            expect = np.tril(Q @ K.T) @ V
            np.testing.assert_allclose(res["out"][t0:t1, h], expect, rtol=1e-12, atol=1e-12)
            # final state is the plain sum of outer products k_s^T v_s
            np.testing.assert_allclose(res["final_state"][b, h, 0], K.T @ V, rtol=1e-12, atol=1e-12)
    assert np.all(res["topk_w"] == 1.0)


@pytest.mark.parametrize("top_k,use_shared,shared_qk", [(1, 1, True), (2, 1, False), (3, 0, True), (4, 1, True)])
def test_recurrence_matches_unrolled_closed_form(top_k, use_shared, shared_qk):
    """The recurrence (eqs. 13-14 + shared) equals the unrolled double sum of
    section 2.4, including an initial state, varlen packing and a query scale."""
    rng = np.random.default_rng(10 + top_k)
    lengths = [9, 1, 0, 23]
    N = 4
    cs = _rand_case(rng, lengths, H=2, c=4, d=3, N=N, shared_qk=shared_qk)
    init = cs["init"] if use_shared else cs["init"][:, :, :N]
    kw = dict(top_k=top_k, use_shared=use_shared, scale=0.7, q_shared=cs["qs"], k_shared=cs["ks"])
    res = oracle.forward(cs["q"], cs["k"], cs["v"], cs["g"], cs["logits"], cs["cu"],
                         initial_state=init, **kw)
    ref = oracle.closed_form(cs["q"], cs["k"], cs["v"], cs["g"], cs["logits"], cs["cu"],
                             initial_state=init, **kw)
    np.testing.assert_allclose(res["out"], ref, rtol=1e-10, atol=1e-10)


def test_unselected_partitions_bitwise_unchanged():
    """Partitions never selected neither decay nor receive writes: their final
    state is bit-identical to the initial state (section 2.2 and eq. 13)."""
    rng = np.random.default_rng(3)
    lengths = [40, 17]
    N = 6
    cs = _rand_case(rng, lengths, H=3, c=4, d=5, N=N)
    logits = cs["logits"].copy()
    logits[..., 4:] = -50.0  # partitions 4 and 5 are never in the top-2
    res = oracle.forward(cs["q"], cs["k"], cs["v"], cs["g"], logits, cs["cu"], top_k=2,
                         initial_state=cs["init"])
    assert np.array_equal(res["final_state"][:, :, 4:6], cs["init"][:, :, 4:6])
    # the selected ones and the shared one did change
    assert not np.array_equal(res["final_state"][:, :, :4], cs["init"][:, :, :4])
    assert not np.array_equal(res["final_state"][:, :, N], cs["init"][:, :, N])
    # decode: per step, every slot outside the selected set and the shared slot is untouched
    state = np.ascontiguousarray(cs["init"][:1].copy())
    for step in range(5):
        before = state.copy()
        tok = rng.normal(size=(1, 3, 4)), rng.random(size=(1, 3, 4)), rng.normal(size=(1, 3, 5)), \
            -rng.random(size=(1, 3, 4)), rng.normal(size=(1, 3, N))
        r = oracle.decode_step(state, *tok, top_k=2)
        for h in range(3):
            chosen = set(r["topk_idx"][0, h].tolist())
            for i in range(N):
                same = np.array_equal(state[0, h, i], before[0, h, i])
                assert same == (i not in chosen)


def test_equal_logits_all_selected_is_scaled_dense_gla():
    """k = N with equal router logits: every partition gets e = 1/N at both
    ends, so the routed output is exactly (1/N) x dense GLA, and the shared
    partition adds one more dense GLA (section 5.3 discussion of k/N = 1)."""
    rng = np.random.default_rng(4)
    lengths = [21, 5]
    N = 4
    cs = _rand_case(rng, lengths, H=2, c=3, d=4, N=N, with_init=False)
    logits = np.zeros_like(cs["logits"])
    gla = oracle.dense_gla(cs["q"], cs["k"], cs["v"], cs["g"], cs["cu"])
    r0 = oracle.forward(cs["q"], cs["k"], cs["v"], cs["g"], logits, cs["cu"], top_k=N, use_shared=0)
    np.testing.assert_allclose(r0["out"], gla / N, rtol=1e-11, atol=1e-12)
    r1 = oracle.forward(cs["q"], cs["k"], cs["v"], cs["g"], logits, cs["cu"], top_k=N, use_shared=1)
    np.testing.assert_allclose(r1["out"], gla * (1 + 1.0 / N), rtol=1e-11, atol=1e-12)


def test_all_selected_general_logits_is_weighted_sum_of_glas():
    """k = N with unequal logits: partition i is a GLA over keys e^i_s k_s read
    with weight e^i_t, so o = sum_i e^i_t GLA(q, e^i k, v, g)_t -- not a single
    state (section 5.3 caution)."""
    rng = np.random.default_rng(5)
    lengths = [19]
    N = 3
    cs = _rand_case(rng, lengths, H=2, c=3, d=2, N=N, with_init=False)
    z = cs["logits"] - cs["logits"].max(-1, keepdims=True)
    e = np.exp(z) / np.exp(z).sum(-1, keepdims=True)
    ref = np.zeros_like(cs["v"])
    for i in range(N):
        ref += e[..., i:i + 1] * oracle.dense_gla(cs["q"], cs["k"] * e[..., i:i + 1], cs["v"], cs["g"], cs["cu"])
    r = oracle.forward(cs["q"], cs["k"], cs["v"], cs["g"], cs["logits"], cs["cu"], top_k=N, use_shared=0)
    np.testing.assert_allclose(r["out"], ref, rtol=1e-11, atol=1e-12)


def test_local_update_clock_worked_example():
    """Page example (section 2.4): retained weight 0.99^100 ~ 0.366 when the
    partition decays at all 100 steps, 0.99^10 ~ 0.904 when it is selected on
    10 of them."""
    with open(os.path.join(GOLDEN, "local_update_clock.json")) as f:
        gold = json.load(f)
    a, span, m = gold["decay_per_step"], gold["span_steps"], gold["active_steps"]
    T = span + 1
    g = np.full((T, 1, 1), np.log(a))
    q = np.ones((T, 1, 1))
    k = np.ones((T, 1, 1))
    v = np.zeros((T, 1, 1))
    v[0] = 1.0
    cu = [0, T]
    # dense: a single partition selected at every step
    dense = oracle.forward(q, k, v, g, np.zeros((T, 1, 1)), cu, top_k=1, use_shared=0)
    ret_dense = dense["out"][span, 0, 0]
    # sparse: partition 0 at t=0 and on m of the following steps, ending at t=span
    active = set(np.linspace(span / m, span, m).round().astype(int).tolist())
    assert len(active) == m and span in active
    logits = np.zeros((T, 1, 2))
    for t in range(T):
        logits[t, 0] = [1.0, 0.0] if (t == 0 or t in active) else [0.0, 1.0]
    sp = oracle.forward(q, k, v, g, logits, cu, top_k=1, use_shared=0)
    e0 = np.exp(1.0) / (np.exp(1.0) + 1.0)
    ret_sparse = sp["out"][span, 0, 0] / (e0 * e0)
    tol = gold["printed_abs_precision"]
    assert abs(ret_dense - gold["printed_retained_every_step"]) < tol
    assert abs(ret_sparse - gold["printed_retained_sparse"]) < tol
    assert ret_dense == pytest.approx(a ** span, rel=1e-12)
    assert ret_sparse == pytest.approx(a ** m, rel=1e-12)


def test_routing_matches_stable_argsort_and_weights_not_renormalised():
    """Top-k indices equal a stable argsort of the negated logits (ties keep
    the lower index); weights are the full-N softmax values, so their sum over
    the selected set is <= 1 (section 2.3 classification-strength identity)."""
    rng = np.random.default_rng(6)
    T, H, N, k = 300, 3, 8, 3
    logits = rng.integers(-2, 3, size=(T, H, N)).astype(np.float64)  # many ties
    cu = [0, 100, 300]
    r = oracle.forward(rng.normal(size=(T, H, 2)), rng.random(size=(T, H, 2)),
                       rng.normal(size=(T, H, 2)), np.zeros((T, H, 2)), logits, cu, top_k=k)
    order = np.argsort(-logits, axis=-1, kind="stable")[..., :k]
    assert np.array_equal(r["topk_idx"], order.astype(np.int32))
    z = np.exp(logits - logits.max(-1, keepdims=True))
    e = z / z.sum(-1, keepdims=True)
    np.testing.assert_allclose(r["topk_w"], np.take_along_axis(e, order, -1), rtol=1e-14)
    assert np.all(r["topk_w"].sum(-1) <= 1.0 + 1e-12)
    assert np.all(r["topk_w"].sum(-1) < 1.0 - 1e-6)  # k < N: strictly below 1


def test_chunk_split_and_decode_continuation():
    """Carrying the state: forward(T) == forward(T1) then forward(T-T1) from its
    final state == forward(T1) then T-T1 decode steps (section 2.6: chunked
    prefill, recurrent decode)."""
    rng = np.random.default_rng(7)
    T, T1, H, c, d, N, k = 30, 11, 2, 4, 3, 5, 2
    cs = _rand_case(rng, [T], H=H, c=c, d=d, N=N)
    a = {n: cs[n] for n in ("q", "k", "v", "g", "logits")}
    full = oracle.forward(*a.values(), [0, T], top_k=k, initial_state=cs["init"])
    first = oracle.forward(*(x[:T1] for x in a.values()), [0, T1], top_k=k, initial_state=cs["init"])
    second = oracle.forward(*(x[T1:] for x in a.values()), [0, T - T1], top_k=k,
                            initial_state=first["final_state"])
    np.testing.assert_allclose(np.concatenate([first["out"], second["out"]]), full["out"], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(second["final_state"], full["final_state"], rtol=1e-12, atol=1e-13)
    state = np.ascontiguousarray(first["final_state"].copy())
    for t in range(T1, T):
        r = oracle.decode_step(state, *(x[t:t + 1] for x in a.values()), top_k=k)
        np.testing.assert_allclose(r["out"][0], full["out"][t], rtol=1e-12, atol=1e-13)
        assert np.array_equal(r["topk_idx"][0], full["topk_idx"][t])
    np.testing.assert_allclose(state, full["final_state"], rtol=1e-12, atol=1e-13)


def test_grouping_is_stable_sort_by_segment():
    """Token->partition grouping (section 2.6): per (sequence, head, partition)
    the tokens in ascending time; equals a lexicographic sort of the routed
    records by (segment, time)."""
    rng = np.random.default_rng(8)
    lengths = [50, 0, 33, 1]
    T, H, N, k = sum(lengths), 3, 6, 2
    cu = np.concatenate([[0], np.cumsum(lengths)])
    logits = rng.integers(-1, 2, size=(T, H, N)).astype(np.float64)
    r = oracle.forward(np.zeros((T, H, 1)), np.zeros((T, H, 1)), np.zeros((T, H, 1)),
                       np.zeros((T, H, 1)), logits, cu, top_k=k, use_shared=0)
    seg_off, perm = oracle.group(r["topk_idx"], cu, N)
    seq_of = np.repeat(np.arange(len(lengths)), lengths)
    t_rec = np.repeat(np.arange(T), H * k)
    h_rec = np.tile(np.repeat(np.arange(H), k), T)
    i_rec = r["topk_idx"].reshape(-1)
    seg_rec = (seq_of[t_rec] * H + h_rec) * N + i_rec
    order = np.lexsort((t_rec, seg_rec))
    assert np.array_equal(perm, t_rec[order])
    counts = np.bincount(seg_rec, minlength=len(lengths) * H * N)
    assert np.array_equal(seg_off, np.concatenate([[0], np.cumsum(counts)]))


def test_generator_blocked_draws_are_identical():
    w = synth.WORKLOADS["tiny_f32"]
    a = synth.make_forward_inputs(w, seed=0)
    b = synth.make_forward_inputs(w, seed=0)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.logits, b.logits)
    rng1, rng2 = np.random.default_rng(0), np.random.default_rng(0)
    x1 = synth._draw(rng1, (37, 2, 3), "bf16", lambda x: x, block_rows=37)
    x2 = synth._draw(rng2, (37, 2, 3), "bf16", lambda x: x, block_rows=5)
    assert np.array_equal(x1, x2)
    # bf16 rounding: round-to-nearest-even of float32
    vals = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e38], dtype=np.float32)
    bits = synth.f32_to_bf16_bits(vals)
    back = synth.bf16_bits_to_f32(bits)
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.015625 and back[3] == -2.5


def test_workload_lengths_seed0():
    w = synth.WORKLOADS["varlen_bf16"]
    rng = np.random.default_rng(0)
    lengths = rng.integers(1024, 32769, 16)
    assert int(lengths.sum()) == 272568
    assert lengths.min() >= 1024 and lengths.max() <= 32768
    assert w.num_slots == 17
