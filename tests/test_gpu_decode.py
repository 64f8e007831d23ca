"""GPU parity of sse_decode_step against the fp64 oracle (marked gpu)."""
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


def _decode_run(w, batch, steps, init_std=0.1, sample=None):
    import oracle
    from sparse_state_linear_router_gb300 import binding
    cfg = H_.config_of(w)
    P = w.num_slots
    rng = np.random.default_rng(77)
    state0 = (rng.normal(size=(batch, w.num_heads, P, w.key_dim, w.value_dim)) * init_std).astype(np.float32)
    sample = np.arange(batch) if sample is None else np.asarray(sample)
    ref_state = np.ascontiguousarray(state0[sample].astype(np.float64))
    dstate = torch.from_numpy(state0).cuda()
    for s in range(steps):
        tok = synth.make_decode_inputs(w, s, batch=batch)
        before = dstate.clone()
        dv = {n: binding.to_device(getattr(tok, n)) for n in ("q", "k", "v", "g", "logits")}
        r = binding.decode_step(cfg, dstate, dv["q"], dv["k"], dv["v"], dv["g"], dv["logits"],
                                want_routing=True)
        torch.cuda.synchronize()
        ref = oracle.decode_step(ref_state, *(getattr(tok, n)[sample] for n in ("q", "k", "v", "g", "logits")),
                                 top_k=w.top_k, use_shared=w.use_shared)
        idx = H_.to_numpy(r["topk_idx"])[sample]
        assert np.array_equal(idx, ref["topk_idx"])
        np.testing.assert_allclose(H_.to_numpy(r["topk_w"])[sample], ref["topk_w"], rtol=2e-6, atol=1e-7)
        assert H_.max_abs_rel(H_.to_numpy(r["out"])[sample], ref["out"]) < H_.tol_for(w)
        assert H_.max_abs_rel(H_.to_numpy(dstate)[sample], ref_state) < H_.tol_for(w)
        # unselected states: bit-identical after the step
        changed = (dstate != before).flatten(3).any(-1).cpu().numpy()  # [B,H,P]
        sel = np.zeros(changed.shape, dtype=bool)
        all_idx = H_.to_numpy(r["topk_idx"])
        np.put_along_axis(sel, all_idx.astype(np.int64), True, axis=-1)
        if w.use_shared:
            sel[..., w.num_partitions] = True
        assert not np.any(changed & ~sel)


def test_decode_small_f32():
    w = H_.workload_variant("decode_bf16", dtype="f32", num_heads=2, key_dim=16, value_dim=16,
                            num_partitions=4, top_k=1)
    _decode_run(w, batch=5, steps=4)


def test_decode_bf16_reduced_batch():
    w = synth.WORKLOADS["decode_bf16"]
    _decode_run(w, batch=4, steps=3)


def test_decode_noshared_k3_d64():
    w = H_.workload_variant("decode_bf16", num_heads=3, key_dim=64, value_dim=64, num_partitions=8,
                            top_k=3, use_shared=0)
    _decode_run(w, batch=6, steps=3)


def test_decode_full_batch_sampled():
    """Full decode workload (256 sequences x 16 heads, N=16): every sequence
    is stepped on the GPU, a sample of sequences is recomputed by the oracle."""
    w = synth.WORKLOADS["decode_bf16"]
    _decode_run(w, batch=w.decode_batch, steps=2, sample=[0, 17, 128, 255])


def test_decode_matches_forward_continuation():
    """forward over T tokens then decode steps == forward over T + steps
    tokens (state carry from the chunked prefill into the recurrent decode)."""
    from sparse_state_linear_router_gb300 import binding
    w = H_.workload_variant("small_bf16", num_heads=2)
    T1, extra = 200, 3
    inp = synth.make_forward_inputs(w, seed=4, lengths=[T1 + extra], with_init=True)
    first = synth.LayerInputs(w, inp.q[:T1], inp.k[:T1], inp.v[:T1], inp.g[:T1], inp.logits[:T1],
                              np.array([0, T1], np.int32), inp.init_state)
    g1 = H_.run_gpu_forward(w, first)
    full = H_.run_oracle_forward(w, inp)
    cfg = H_.config_of(w)
    st = torch.from_numpy(np.ascontiguousarray(g1["final_state"])).cuda()
    for t in range(T1, T1 + extra):
        dv = {n: binding.to_device(np.ascontiguousarray(getattr(inp, n)[t:t + 1])) for n in ("q", "k", "v", "g", "logits")}
        r = binding.decode_step(cfg, st, dv["q"], dv["k"], dv["v"], dv["g"], dv["logits"])
        torch.cuda.synchronize()
        assert H_.max_abs_rel(H_.to_numpy(r["out"])[0], full["out"][t]) < H_.TOL_BF16
    assert H_.max_abs_rel(H_.to_numpy(st), full["final_state"]) < H_.TOL_BF16


def test_decode_1000_steps_full_size():
    """The full decode workload run for 1000 consecutive steps on states
    resident in device memory: 256 sequences x 16 heads, N = 16 routed
    partitions of 128 x 128 plus the shared one (4.6 GB of float32 states),
    fresh seeded inputs every step (seed 1000 + s).  The fp64 oracle follows a
    sample of sequences (first, middle, last and two others) through every
    step; routing is compared bit for bit every step, outputs and states at
    steps 0, 1, 499 and 999 (float32 drift of the in-place updates would show
    there); every step, every state the step did not select must be
    bit-identical to before the step ("Scaling Linear Attention with Sparse
    State Expansion", section 2.6: decoding recurs only on the selected
    states)."""
    import concurrent.futures as cf

    import oracle
    from sparse_state_linear_router_gb300 import binding
    w = synth.WORKLOADS["decode_bf16"]
    B, H, N, P = w.decode_batch, w.num_heads, w.num_partitions, w.num_slots
    steps, checkpoints = 1000, {0, 1, 499, 999}
    sample = np.array([0, 61, 128, 200, B - 1])
    cfg = H_.config_of(w)
    dstate = torch.zeros((B, H, P, w.key_dim, w.value_dim), dtype=torch.float32, device="cuda")
    before = torch.empty_like(dstate)
    ref_state = np.zeros((len(sample), H, P, w.key_dim, w.value_dim), dtype=np.float64)
    checked = []
    # the inputs of later steps are drawn on host threads while the GPU and the
    # oracle work on the current one (numpy's generators and ufuncs release the GIL)
    with cf.ThreadPoolExecutor(max_workers=8) as pool:
        futs = {s: pool.submit(synth.make_decode_inputs, w, s, B) for s in range(min(steps, 16))}
        for s in range(steps):
            tok = futs.pop(s).result()
            if s + 16 < steps:
                futs[s + 16] = pool.submit(synth.make_decode_inputs, w, s + 16, B)
            before.copy_(dstate)
            dv = {n: binding.to_device(getattr(tok, n)) for n in ("q", "k", "v", "g", "logits")}
            r = binding.decode_step(cfg, dstate, dv["q"], dv["k"], dv["v"], dv["g"], dv["logits"],
                                    want_routing=True)
            ref = oracle.decode_step(ref_state, *(getattr(tok, n)[sample] for n in ("q", "k", "v", "g", "logits")),
                                     top_k=w.top_k, use_shared=w.use_shared)
            all_idx = H_.to_numpy(r["topk_idx"])
            assert np.array_equal(all_idx[sample], ref["topk_idx"]), s
            # states the step did not select: bit-identical
            changed = (dstate != before).flatten(3).any(-1).cpu().numpy()  # [B, H, P]
            sel = np.zeros(changed.shape, dtype=bool)
            np.put_along_axis(sel, all_idx.astype(np.int64), True, axis=-1)
            sel[..., N] = True
            assert not np.any(changed & ~sel), s
            if s in checkpoints:
                e_out = H_.max_abs_rel(H_.to_numpy(r["out"])[sample], ref["out"])
                e_st = H_.max_abs_rel(H_.to_numpy(dstate[torch.from_numpy(sample).cuda()]), ref_state)
                checked.append((s, e_out, e_st))
                assert e_out < H_.TOL_BF16 and e_st < H_.TOL_BF16, (s, e_out, e_st)
    assert [c[0] for c in checked] == sorted(checkpoints)
    print("decode 1000 steps: (step, out err, state err)", checked)
