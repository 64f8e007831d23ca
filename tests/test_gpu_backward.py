"""GPU parity of sse_backward against the float64 backward oracle
(``oracle/backward.py``, itself pinned by finite differences of the forward
oracle), on the same seeded inputs, through the C ABI (marked gpu).

The GPU side takes the gate gradient through the running sum of the log-gate
(dL/dG_t = Q_t * u_t - K_t * dK_t, reverse-summed); the oracle takes it
through the decay of every step (rowsum(G * S_before) * a): two different
routes to the same number."""
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


def _store(x, dtype):
    x = np.asarray(x, dtype=np.float32)
    return x if dtype == "f32" else synth.f32_to_bf16_bits(x)


def _run(w, inp, *, seed=0, with_dfin=True, separate_shared=False, scale=1.0, pairs_only=None, algo="auto"):
    """GPU and oracle gradients of <d_out, out> + <d_final, final_state>."""
    from oracle import backward as bw
    from sparse_state_linear_router_gb300 import binding
    rng = np.random.default_rng(100 + seed)
    T, S, H = inp.total_tokens, inp.num_seqs, w.num_heads
    P = w.num_slots
    d_out = _store(rng.normal(size=(T, H, w.value_dim)), w.dtype)
    d_fin = (rng.normal(size=(S, H, P, w.key_dim, w.value_dim)) * 0.5).astype(np.float32) if with_dfin else None
    qs = ks = None
    if separate_shared:
        qs = _store(rng.normal(size=inp.q.shape) / np.sqrt(w.key_dim), w.dtype)
        ks = _store(rng.random(size=inp.k.shape) / w.key_dim, w.dtype)
    cfg = H_.config_of(w, algo=algo, scale=scale)
    dv_ = lambda a: None if a is None else binding.to_device(a)  # noqa: E731
    t = {n: dv_(getattr(inp, n)) for n in ("q", "k", "v", "g", "logits")}
    cu = torch.from_numpy(inp.cu_seqlens).cuda()
    init = None if inp.init_state is None else torch.from_numpy(inp.init_state).cuda()
    dfin_t = None if d_fin is None else torch.from_numpy(d_fin).cuda()
    r = binding.backward(cfg, t["q"], t["k"], t["v"], t["g"], t["logits"], cu, dv_(d_out), q_shared=dv_(qs),
                         k_shared=dv_(ks), initial_state=init, d_final_state=dfin_t)
    torch.cuda.synchronize()
    gpu = {k_: (None if v_ is None else H_.to_numpy(v_)) for k_, v_ in r.items() if k_ != "workspace"}
    if pairs_only is None:
        ref = bw.backward(inp.q, inp.k, inp.v, inp.g, inp.logits, inp.cu_seqlens, d_out, top_k=w.top_k,
                          use_shared=w.use_shared, scale=scale, q_shared=qs, k_shared=ks,
                          initial_state=inp.init_state, d_final_state=d_fin)
        return gpu, ref, None
    # one (sequence, head) pair at a time: the gradients of a pair depend on its own rows only
    refs = []
    for p in pairs_only:
        b, h = divmod(int(p), H)
        t0, t1 = int(inp.cu_seqlens[b]), int(inp.cu_seqlens[b + 1])
        sl = lambda a: None if a is None else np.ascontiguousarray(a[t0:t1, h:h + 1])  # noqa: E731
        ref = bw.backward(sl(inp.q), sl(inp.k), sl(inp.v), sl(inp.g), sl(inp.logits),
                          np.array([0, t1 - t0]), sl(d_out), top_k=w.top_k, use_shared=w.use_shared, scale=scale,
                          q_shared=sl(qs), k_shared=sl(ks),
                          initial_state=None if inp.init_state is None else inp.init_state[b:b + 1, h:h + 1],
                          d_final_state=None if d_fin is None else d_fin[b:b + 1, h:h + 1])
        refs.append((b, h, t0, t1, ref))
    return gpu, None, refs


NAMES = ("dq", "dk", "dv", "dg", "dlogits", "d_initial_state", "dq_shared", "dk_shared")


def _compare(gpu, ref, tol):
    for n in NAMES:
        if ref[n] is None:
            assert gpu[n] is None, n
            continue
        err = H_.max_abs_rel(gpu[n], ref[n])
        assert err < tol, (n, err)


CASES = {
    # name: (workload, lengths, overrides, kwargs)
    "tiny_f32": ("tiny_f32", [40, 0, 23], {}, {}),
    "f32_separate_shared": ("tiny_f32", [31, 17], {"num_partitions": 4, "top_k": 2}, {"separate_shared": True}),
    "small_bf16_varlen": ("small_bf16", [300, 1, 0, 129], {"num_heads": 2}, {}),
    "bf16_scale_separate_shared": ("small_bf16", [200, 77], {"num_heads": 2}, {"separate_shared": True, "scale": 0.5}),
    "noshared_k3": ("small_bf16", [180], {"num_heads": 1, "num_partitions": 6, "top_k": 3, "use_shared": 0}, {}),
    "k_equals_N": ("small_bf16", [150, 60], {"num_heads": 1, "num_partitions": 3, "top_k": 3}, {}),
    "c128_d128_no_dfin": ("layer_bf16", [257, 64], {"num_heads": 1, "num_partitions": 4}, {"with_dfin": False}),
    "c128_d64": ("layer_bf16", [130, 3], {"num_heads": 2, "value_dim": 64}, {}),
    "c128_noshared_k3": ("layer_bf16", [260, 1, 0], {"num_heads": 2, "num_partitions": 6, "top_k": 3,
                                                     "use_shared": 0}, {}),
    "c128_k_equals_N": ("layer_bf16", [200, 57], {"num_heads": 1, "num_partitions": 3, "top_k": 3}, {"scale": 0.5}),
}


def _algos(w):
    """The chunked (tensor-core) form where it applies (bf16, c = 128), and the
    per-token one everywhere."""
    return ["recurrent", "chunked"] if (w.dtype == "bf16" and w.key_dim == 128) else ["recurrent"]


@pytest.mark.parametrize("name", sorted(CASES))
def test_backward_matches_oracle(name):
    wname, lengths, over, kw = CASES[name]
    w = H_.workload_variant(wname, **over)
    inp = synth.make_forward_inputs(w, seed=3, lengths=lengths, with_init=True)
    for algo in _algos(w):
        gpu, ref, _ = _run(w, inp, algo=algo, **kw)
        _compare(gpu, ref, H_.tol_for(w))


@pytest.mark.parametrize("dv", [128, 64])
def test_backward_chunked_many_chunks(dv):
    """Segments of several chunks with ragged tails, empty sequences and
    separate shared q / k: the chunked form's scan over chunks and its
    suffix sums of the gate gradient carry across chunk boundaries."""
    w = H_.workload_variant("layer_bf16", num_heads=2, num_partitions=4, top_k=2, value_dim=dv)
    inp = synth.make_forward_inputs(w, seed=21, lengths=[700, 0, 300, 129], with_init=True)
    gpu, ref, _ = _run(w, inp, algo="chunked", separate_shared=True, scale=0.75)
    _compare(gpu, ref, H_.TOL_BF16)


def test_backward_chunked_strong_gates():
    """Log-gates of -5 on a run of rows push some chunks past the factorised
    form's range (|G_m| or |G_l - G_m| > 64): those work items go to the
    per-token kernel, the rest stay chunked, and every gradient matches."""
    w = H_.workload_variant("layer_bf16", num_heads=2, num_partitions=4, top_k=2)
    inp = synth.make_forward_inputs(w, seed=5, lengths=[400, 260], with_init=True)
    g = synth.bf16_bits_to_f32(inp.g)
    g[100:180, 0] = -5.0       # shared and routed segments of head 0 in sequence 0
    g[500:520, 1] = -3.0       # a milder run in sequence 1, head 1
    inp.g = synth.f32_to_bf16_bits(g.astype(np.float32))
    gpu, ref, _ = _run(w, inp, algo="chunked")
    _compare(gpu, ref, H_.TOL_BF16)


def test_backward_skewed_routing_and_empty_segments():
    """Per-partition router bias: some partitions take nearly every token,
    others none, so empty segments (whose initial-state gradient is the final
    state's gradient, undecayed) meet long ones."""
    w = H_.workload_variant("small_bf16", num_heads=2, num_partitions=8, top_k=2)
    inp = synth.make_forward_inputs(w, seed=12, lengths=[260, 0, 41], with_init=True)
    beta = 8.0 * (np.arange(8) / 7 - 0.5) * 2.0
    inp.logits = synth.f32_to_bf16_bits((synth.bf16_bits_to_f32(inp.logits) + beta).astype(np.float32))
    gpu, ref, _ = _run(w, inp)
    _compare(gpu, ref, H_.TOL_BF16)


def test_backward_layer_shape_sampled_pairs():
    """The layer workload's shape (16 heads, c = d = 128, N = 8, top-2,
    shared, 8 sequences) at 256 tokens per sequence through the GPU backward;
    the oracle -- which keeps every state, 2.4 MB per token here -- recomputes
    three (sequence, head) pairs on their own rows."""
    w = synth.WORKLOADS["layer_bf16"]
    inp = synth.make_forward_inputs(w, seed=0, lengths=[256] * 8, with_init=True)
    S, H = inp.num_seqs, w.num_heads
    pairs = [0, 37, S * H - 1]
    gpu, _, refs = _run(w, inp, pairs_only=pairs)
    for b, h, t0, t1, ref in refs:
        for n in ("dq", "dk", "dv", "dg", "dlogits"):
            err = H_.max_abs_rel(gpu[n][t0:t1, h:h + 1], ref[n])
            assert err < H_.TOL_BF16, (b, h, n, err)
        err = H_.max_abs_rel(gpu["d_initial_state"][b:b + 1, h:h + 1], ref["d_initial_state"])
        assert err < H_.TOL_BF16, (b, h, "d_initial_state", err)


@pytest.mark.parametrize("half", [1024, 4096])
def test_backward_fig6_shape_sampled_pairs(half):
    """Fig. 6's operator shape ("Scaling Linear Attention with Sparse State
    Expansion", section 2.6: 8 heads, head dim 128, top-1 of N = 4, shared,
    cu_seqlens = [0, L/2, L]) at L = 2048 (256 chunks, more than the chunked
    kernels' persistent CTAs, so each of them walks several chunks) and at the
    benchmark's L = 8192.  The oracle recomputes a few (sequence, head) pairs
    on their own rows."""
    w = H_.workload_variant("layer_bf16", num_heads=8, num_partitions=4, top_k=1)
    inp = synth.make_forward_inputs(w, seed=6, lengths=[half, half], with_init=True)
    S, H = inp.num_seqs, w.num_heads
    pairs = [0, 11, S * H - 1] if half <= 1024 else [3, S * H - 1]
    gpu, _, refs = _run(w, inp, pairs_only=pairs, algo="chunked")
    for b, h, t0, t1, ref in refs:
        for n in ("dq", "dk", "dv", "dg", "dlogits"):
            err = H_.max_abs_rel(gpu[n][t0:t1, h:h + 1], ref[n])
            assert err < H_.TOL_BF16, (b, h, n, err)
        err = H_.max_abs_rel(gpu["d_initial_state"][b:b + 1, h:h + 1], ref["d_initial_state"])
        assert err < H_.TOL_BF16, (b, h, "d_initial_state", err)


def test_backward_chunked_without_initial_state():
    """No initial state and no final-state gradient (the usual training call):
    the scan starts from zero states, the gate gradient's final term is zero,
    and d_initial_state is the gradient of a zero initial state."""
    w = H_.workload_variant("layer_bf16", num_heads=2, num_partitions=4, top_k=2)
    inp = synth.make_forward_inputs(w, seed=8, lengths=[333, 0, 140], with_init=False)
    gpu, ref, _ = _run(w, inp, algo="chunked", with_dfin=False)
    _compare(gpu, ref, H_.TOL_BF16)


def test_backward_varlen_full_size_chunked_matches_per_token():
    """The long-context varlen workload at full size (16 packed sequences of
    1024-32768 tokens, 16 heads, c = d = 128, N = 16, top-2, shared, random
    initial state; about 110 000 chunks): every gradient of the chunked form
    against the per-token form on the same inputs.  Each is within bf16
    rounding of the exact result (the parity cases above), so they agree to
    the same tolerance."""
    from sparse_state_linear_router_gb300 import binding
    w = synth.WORKLOADS["varlen_bf16"]
    x = synth.make_forward_inputs_device(w, seed=0)
    T, S, H = x["total_tokens"], x["num_seqs"], w.num_heads
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    d_out = torch.randn((T, H, w.value_dim), generator=gen, device="cuda").to(torch.bfloat16)
    d_fin = torch.randn((S, H, w.num_slots, w.key_dim, w.value_dim), generator=gen, device="cuda") * 0.5
    res = {}
    for algo in ("chunked", "recurrent"):
        cfg = H_.config_of(w, algo)
        r = binding.backward(cfg, x["q"], x["k"], x["v"], x["g"], x["logits"], x["cu_seqlens"], d_out,
                             initial_state=x["init"], d_final_state=d_fin)
        torch.cuda.synchronize()
        res[algo] = {n: v for n, v in r.items() if n != "workspace" and v is not None}
        del r
        torch.cuda.empty_cache()
    for n in res["chunked"]:
        a, b = res["chunked"][n].float(), res["recurrent"][n].float()
        assert bool(torch.isfinite(a).all()), n
        err = float((a - b).abs().max() / b.abs().max().clamp_min(1e-6))
        assert err < H_.TOL_BF16, (n, err)
