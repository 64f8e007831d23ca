"""GPU parity of SSE on the gated delta rule (sse_delta_forward,
sse_delta_decode_step) against the float64 oracle ``oracle/delta.py`` on the
same seeded inputs, through the C ABI (marked gpu)."""
import numpy as np
import pytest

from sparse_state_linear_router_gb300 import inputs as synth
from tests import _helpers as H_

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_state_linear_router_gb300 import binding
    binding.load()


def _gpu(w, inp, scale=1.0, qs=None, ks=None, algo="auto"):
    from sparse_state_linear_router_gb300 import binding
    cfg = H_.config_of(w, algo, scale=scale)
    t = {n: binding.to_device(getattr(inp, n)) for n in ("q", "k", "v", "log_alpha", "beta", "logits")}
    cu = torch.from_numpy(inp.cu_seqlens).cuda()
    init = None if inp.init_state is None else torch.from_numpy(inp.init_state).cuda()
    dv = lambda a: None if a is None else binding.to_device(a)  # noqa: E731
    r = binding.delta_forward(cfg, t["q"], t["k"], t["v"], t["log_alpha"], t["beta"], t["logits"], cu,
                              q_shared=dv(qs), k_shared=dv(ks), initial_state=init, want_routing=True)
    torch.cuda.synchronize()
    return {n: H_.to_numpy(r[n]) for n in ("out", "final_state", "topk_idx", "topk_w")}


def _ref(w, inp, scale=1.0, qs=None, ks=None):
    from oracle import delta as dl
    return dl.delta_forward(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.logits, inp.cu_seqlens,
                            top_k=w.top_k, use_shared=w.use_shared, scale=scale, q_shared=qs, k_shared=ks,
                            initial_state=inp.init_state)


CASES = {
    "tiny_f32": ("tiny_f32", [40, 0, 23], {}),
    "f32_d64": ("tiny_f32", [37, 20], {"key_dim": 64, "value_dim": 64, "num_partitions": 8, "top_k": 2}),
    "small_bf16": ("small_bf16", [300, 1, 0, 129], {"num_heads": 2}),
    "noshared_k3": ("small_bf16", [180], {"num_heads": 1, "num_partitions": 6, "top_k": 3, "use_shared": 0}),
    "c128_d128": ("layer_bf16", [257, 64], {"num_heads": 2}),
    "c128_d64": ("layer_bf16", [130, 3], {"num_heads": 2, "value_dim": 64}),
    # segments of hundreds of rows: many 32-row record blocks and wraps of the
    # row pipeline of the c = 128 kernel
    "c128_long": ("layer_bf16", [1500, 0, 700], {"num_heads": 1, "num_partitions": 4, "top_k": 1}),
    "c128_d64_long": ("layer_bf16", [901], {"num_heads": 1, "value_dim": 64, "num_partitions": 2, "top_k": 1}),
    # one sequence of the layer shape's length: 32 chunks carry the state
    "c128_4096": ("layer_bf16", [4096], {"num_heads": 1, "num_partitions": 4, "top_k": 1}),
}


def _algos(name):
    """Both forms where the chunked tensor-core one applies (bf16, c = d = 128):
    auto takes it, recurrent keeps the token-serial kernel."""
    wname, _, over = CASES[name]
    w = H_.workload_variant(wname, **over)
    if w.dtype == "bf16" and w.key_dim == 128 and w.value_dim == 128:
        return ["auto", "recurrent"]
    return ["auto"]


@pytest.mark.parametrize("name,algo", [(n, a) for n in sorted(CASES) for a in _algos(n)])
def test_delta_forward_matches_oracle(name, algo):
    wname, lengths, over = CASES[name]
    w = H_.workload_variant(wname, **over)
    inp = synth.make_delta_inputs(w, seed=4, lengths=lengths, with_init=True)
    gpu, ref = _gpu(w, inp, algo=algo), _ref(w, inp)
    assert np.array_equal(gpu["topk_idx"], ref["topk_idx"])
    tol = H_.tol_for(w)
    assert H_.max_abs_rel(gpu["out"], ref["out"]) < tol
    assert H_.max_abs_rel(gpu["final_state"], ref["final_state"]) < tol


def test_delta_full_size_sampled_pairs():
    """The layer shape the benchmark times (8 x 4096 tokens, H16, c = d = 128,
    N8, top-2, shared, random initial states) in one call of the chunked form;
    the oracle recomputes a sample of (sequence, head) pairs, each from its own
    slice of the inputs (heads and sequences are independent), and the routing
    of those rows is compared exactly."""
    import dataclasses
    w = synth.WORKLOADS["layer_bf16"]
    inp = synth.make_delta_inputs(w, seed=11, with_init=True)
    gpu = _gpu(w, inp)
    S, H = len(inp.cu_seqlens) - 1, w.num_heads
    rng = np.random.default_rng(321)
    pairs = sorted(set(rng.choice(S * H, size=3, replace=False).tolist()) | {S * H - 1})
    for p in pairs:
        b, h = divmod(int(p), H)
        t0, t1 = int(inp.cu_seqlens[b]), int(inp.cu_seqlens[b + 1])
        sub = dataclasses.replace(
            inp, q=inp.q[t0:t1, h:h + 1], k=inp.k[t0:t1, h:h + 1], v=inp.v[t0:t1, h:h + 1],
            log_alpha=inp.log_alpha[t0:t1, h:h + 1], beta=inp.beta[t0:t1, h:h + 1],
            logits=inp.logits[t0:t1, h:h + 1], cu_seqlens=np.array([0, t1 - t0], dtype=np.int32),
            init_state=inp.init_state[b:b + 1, h:h + 1])
        ref = _ref(w, sub)
        assert np.array_equal(gpu["topk_idx"][t0:t1, h], ref["topk_idx"][:, 0])
        assert H_.max_abs_rel(gpu["out"][t0:t1, h], ref["out"][:, 0]) < H_.TOL_BF16
        assert H_.max_abs_rel(gpu["final_state"][b, h], ref["final_state"][0, 0]) < H_.TOL_BF16


@pytest.mark.parametrize("algo", ["auto", "recurrent"])
def test_delta_forward_strong_and_mild_decay(algo):
    """Chunks whose summed log-decay spans more than 60 either side of their
    midpoint (log-gates of -1.5 on every row of the first 300 tokens) beside
    chunks of the mild recipe: the chunked form forms their decay factors one
    element at a time, the others around the midpoint; both must match."""
    w = H_.workload_variant("layer_bf16", num_heads=2, num_partitions=4, top_k=1)
    inp = synth.make_delta_inputs(w, seed=8, lengths=[700, 260], with_init=True)
    la = synth.bf16_bits_to_f32(inp.log_alpha)
    la[:300] = -1.5
    la[760:800] = -4.0
    inp.log_alpha = synth.f32_to_bf16_bits(la)
    gpu, ref = _gpu(w, inp, algo=algo), _ref(w, inp)
    assert np.array_equal(gpu["topk_idx"], ref["topk_idx"])
    assert H_.max_abs_rel(gpu["out"], ref["out"]) < H_.TOL_BF16
    assert H_.max_abs_rel(gpu["final_state"], ref["final_state"]) < H_.TOL_BF16


@pytest.mark.parametrize("wname,over,algo", [("small_bf16", {"num_heads": 2}, "auto"),
                                             ("layer_bf16", {"num_heads": 1}, "auto"),
                                             ("layer_bf16", {"num_heads": 1}, "recurrent")])
def test_delta_scale_separate_shared_and_untouched_states(wname, over, algo):
    w = H_.workload_variant(wname, num_partitions=6, top_k=2, **over)
    inp = synth.make_delta_inputs(w, seed=5, lengths=[200, 41], with_init=True)
    inp.logits[..., 4:] = synth.f32_to_bf16_bits(np.full(inp.logits[..., 4:].shape, -60.0, np.float32))
    rng = np.random.default_rng(6)
    qs = synth.f32_to_bf16_bits((rng.normal(size=inp.q.shape) / 8).astype(np.float32))
    ks = synth.f32_to_bf16_bits((rng.normal(size=inp.k.shape) / 11).astype(np.float32))
    gpu, ref = _gpu(w, inp, 0.6, qs, ks, algo=algo), _ref(w, inp, 0.6, qs, ks)
    assert H_.max_abs_rel(gpu["out"], ref["out"]) < H_.TOL_BF16
    assert H_.max_abs_rel(gpu["final_state"], ref["final_state"]) < H_.TOL_BF16
    assert np.array_equal(gpu["final_state"][:, :, 4:6], inp.init_state[:, :, 4:6])


@pytest.mark.parametrize("wname,over", [("tiny_f32", {}), ("layer_bf16", {"num_heads": 2, "num_partitions": 8})])
def test_delta_decode_continues_the_forward(wname, over):
    """Forward over the first tokens, then decode steps on the resident
    states: each step matches the oracle's decode, the unselected states stay
    bit for bit, and the end equals the oracle's forward over all tokens."""
    from oracle import delta as dl
    from sparse_state_linear_router_gb300 import binding
    w = H_.workload_variant(wname, **over)
    T1, extra, B = 40, 4, 3
    inp = synth.make_delta_inputs(w, seed=7, lengths=[T1 + extra] * B, with_init=True)
    cfg = H_.config_of(w)
    cu = inp.cu_seqlens
    # forward over the first T1 tokens of every sequence
    sel = np.concatenate([np.arange(cu[b], cu[b] + T1) for b in range(B)])
    head = synth.DeltaInputs(w, inp.q[sel], inp.k[sel], inp.v[sel], inp.log_alpha[sel], inp.beta[sel],
                             inp.logits[sel], np.arange(B + 1, dtype=np.int32) * T1, inp.init_state)
    st = torch.from_numpy(np.ascontiguousarray(_gpu(w, head)["final_state"])).cuda()
    ref_state = np.ascontiguousarray(_ref(w, head)["final_state"])
    tol = H_.tol_for(w)
    for s in range(extra):
        rows = cu[:-1] + T1 + s
        x = {n: binding.to_device(np.ascontiguousarray(getattr(inp, n)[rows]))
             for n in ("q", "k", "v", "log_alpha", "beta", "logits")}
        before = st.clone()
        r = binding.delta_decode_step(cfg, st, x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["logits"],
                                      want_routing=True)
        torch.cuda.synchronize()
        ref = dl.delta_decode_step(ref_state, *(getattr(inp, n)[rows] for n in ("q", "k", "v", "log_alpha", "beta",
                                                                               "logits")),
                                   top_k=w.top_k, use_shared=w.use_shared)
        idx = H_.to_numpy(r["topk_idx"])
        assert np.array_equal(idx, ref["topk_idx"])
        assert H_.max_abs_rel(H_.to_numpy(r["out"]), ref["out"]) < tol
        changed = (st != before).flatten(3).any(-1).cpu().numpy()
        chosen = np.zeros(changed.shape, dtype=bool)
        np.put_along_axis(chosen, idx.astype(np.int64), True, axis=-1)
        chosen[..., w.num_partitions] = True
        assert not np.any(changed & ~chosen)
    full = _ref(w, inp)
    assert H_.max_abs_rel(H_.to_numpy(st), full["final_state"]) < tol
