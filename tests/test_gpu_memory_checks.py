"""Memory-behaviour checks of the CUDA path (marked gpu): stand-ins for a
sanitizer on a pool where compute-sanitizer is closed.

* Guard regions: every output of sse_forward (each schedule), sse_decode_step
  and sse_front_end is placed inside a larger buffer whose bytes before and
  after it hold a canary pattern; after the call the canaries must be intact
  (no write outside an output) and the outputs equal to a plain call's.
* Poisoned workspace: the workspace is filled with 0xFF bytes (NaN floats,
  -1 integers) before the call; the outputs must be bit-identical to a call
  on a zero-filled workspace (nothing reads workspace memory it did not write).
* State carry (checkpoint / resume): forward over the first T1 tokens, then
  over the rest with the first call's final state as the initial state, equals
  one forward over all tokens (the method's only sequential dependency).
"""
import numpy as np
import pytest

from sparse_state_linear_router_gb300 import inputs as synth
from tests import _helpers as H_

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

CANARY = 0x5A
GUARD = 4096  # bytes on each side of an output


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_state_linear_router_gb300 import binding
    binding.load()


def _guarded(shape, dtype):
    """A tensor of `shape` inside a canary-filled byte buffer; returns (view, raw)."""
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    raw = torch.full((GUARD + n + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
    view = raw[GUARD:GUARD + n].view(dtype).view(*shape)
    view.zero_()
    return view, raw


def _canaries_intact(raw, n):
    host = raw.cpu().numpy()
    return bool(np.all(host[:GUARD] == CANARY) and np.all(host[GUARD + n:] == CANARY))


def _fwd_case():
    w = H_.workload_variant("layer_bf16", num_heads=2)
    inp = synth.make_forward_inputs(w, seed=9, lengths=[300, 1, 0, 517], with_init=True)
    return w, inp


def _fwd_call(w, inp, algo, out=None, final_state=None, workspace=None):
    from sparse_state_linear_router_gb300 import binding
    cfg = H_.config_of(w, algo)
    t = {n: binding.to_device(getattr(inp, n)) for n in ("q", "k", "v", "g", "logits")}
    cu = torch.from_numpy(inp.cu_seqlens.astype(np.int32)).cuda()
    init = torch.from_numpy(inp.init_state).cuda()
    res = binding.forward(cfg, t["q"], t["k"], t["v"], t["g"], t["logits"], cu, initial_state=init, out=out,
                          final_state=final_state, workspace=workspace)
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("algo", ["chunked", "masked", "recurrent"])
def test_forward_writes_only_its_outputs(algo):
    w, inp = _fwd_case()
    ref = _fwd_call(w, inp, algo)
    out, raw_o = _guarded(tuple(ref["out"].shape), ref["out"].dtype)
    fin, raw_f = _guarded(tuple(ref["final_state"].shape), torch.float32)
    res = _fwd_call(w, inp, algo, out=out, final_state=fin)
    assert _canaries_intact(raw_o, out.numel() * out.element_size())
    assert _canaries_intact(raw_f, fin.numel() * 4)
    assert torch.equal(res["out"], ref["out"]) and torch.equal(res["final_state"], ref["final_state"])


@pytest.mark.parametrize("algo", ["chunked", "masked", "recurrent"])
def test_forward_ignores_workspace_contents(algo):
    from sparse_state_linear_router_gb300 import binding
    w, inp = _fwd_case()
    T, S = inp.q.shape[0], len(inp.cu_seqlens) - 1
    ws_zero = binding.forward_workspace(H_.config_of(w, algo), T, S)
    ws_zero.zero_()
    a = _fwd_call(w, inp, algo, workspace=ws_zero)
    ws_poison = torch.full_like(ws_zero, 0xFF)
    b = _fwd_call(w, inp, algo, workspace=ws_poison)
    assert torch.equal(a["out"], b["out"]) and torch.equal(a["final_state"], b["final_state"])


def test_decode_writes_only_its_outputs():
    from sparse_state_linear_router_gb300 import binding
    w = synth.WORKLOADS["decode_bf16"]
    B = 8
    cfg = H_.config_of(w)
    tok = synth.make_decode_inputs(w, 3, batch=B)
    dv = {n: binding.to_device(getattr(tok, n)) for n in ("q", "k", "v", "g", "logits")}
    rng = np.random.default_rng(5)
    s0 = torch.from_numpy((rng.normal(size=(B, w.num_heads, w.num_slots, w.key_dim, w.value_dim)) * 0.1)
                          .astype(np.float32)).cuda()
    st_ref = s0.clone()
    ref = binding.decode_step(cfg, st_ref, dv["q"], dv["k"], dv["v"], dv["g"], dv["logits"])
    st, raw_s = _guarded(tuple(s0.shape), torch.float32)
    st.copy_(s0)
    out, raw_o = _guarded((B, w.num_heads, w.value_dim), torch.bfloat16)
    binding.decode_step(cfg, st, dv["q"], dv["k"], dv["v"], dv["g"], dv["logits"], out=out)
    torch.cuda.synchronize()
    assert _canaries_intact(raw_s, st.numel() * 4) and _canaries_intact(raw_o, out.numel() * 2)
    assert torch.equal(st, st_ref) and torch.equal(out, ref["out"])


def test_front_end_writes_only_its_outputs_and_ignores_workspace():
    from sparse_state_linear_router_gb300 import binding
    w = synth.FRONT_END_WORKLOADS["front_end_small"]
    inp = synth.make_front_end_inputs(w, seed=2)
    cfg = binding.make_config(w.num_heads, w.key_dim, w.value_dim, w.num_partitions, 2, 1, 1.0, "bf16")
    d_ = {n: binding.to_device(getattr(inp, n)) for n in ("x", "w_q", "w_k", "w_v", "w_g", "w_e", "a_q", "b_q",
                                                          "a_k", "b_k")}

    def call(outs=None, workspace=None):
        r = binding.front_end(cfg, d_["x"], d_["w_q"], d_["w_k"], d_["w_v"], d_["w_g"], d_["w_e"], a_q=d_["a_q"],
                              b_q=d_["b_q"], a_k=d_["a_k"], b_k=d_["b_k"], outs=outs, workspace=workspace)
        torch.cuda.synchronize()
        return r

    ref = call()
    names = ("q", "k", "v", "log_gate", "logits", "q_shared", "k_shared")
    guarded = {n: _guarded(tuple(ref[n].shape), torch.bfloat16) for n in names}
    ws = torch.full_like(ref["workspace"], 0xFF)
    ws[:256] = 0
    res = call(outs={n: guarded[n][0] for n in names}, workspace=ws)
    for n in names:
        view, raw = guarded[n]
        assert _canaries_intact(raw, view.numel() * 2), n
        assert torch.equal(res[n], ref[n]), n


@pytest.mark.parametrize("algo", ["chunked", "recurrent"])
def test_forward_state_carry_split(algo):
    """forward(all) == forward(first T1 tokens) then forward(rest) from its final state."""
    from sparse_state_linear_router_gb300 import binding
    w = H_.workload_variant("layer_bf16", num_heads=2)
    L = 700
    full = synth.make_forward_inputs(w, seed=12, lengths=[L], with_init=True)
    cfg = H_.config_of(w, algo)
    t = {n: binding.to_device(getattr(full, n)) for n in ("q", "k", "v", "g", "logits")}
    init = torch.from_numpy(full.init_state).cuda()
    for T1 in (256, 333):
        a = binding.forward(cfg, *(t[n] for n in ("q", "k", "v", "g", "logits")),
                            torch.tensor([0, L], dtype=torch.int32, device="cuda"), initial_state=init)
        p1 = binding.forward(cfg, *(t[n][:T1] for n in ("q", "k", "v", "g", "logits")),
                             torch.tensor([0, T1], dtype=torch.int32, device="cuda"), initial_state=init)
        p2 = binding.forward(cfg, *(t[n][T1:].contiguous() for n in ("q", "k", "v", "g", "logits")),
                             torch.tensor([0, L - T1], dtype=torch.int32, device="cuda"),
                             initial_state=p1["final_state"])
        torch.cuda.synchronize()
        both = torch.cat([p1["out"], p2["out"]])
        assert H_.max_abs_rel(H_.to_numpy(both), H_.to_numpy(a["out"])) < H_.TOL_BF16
        # the two runs cut the sequence into different chunks (bf16 operands)
        assert H_.max_abs_rel(H_.to_numpy(p2["final_state"]), H_.to_numpy(a["final_state"])) < H_.TOL_BF16


@pytest.mark.parametrize("algo,dv", [("chunked", 128), ("chunked", 64), ("recurrent", 128)])
def test_backward_writes_only_its_outputs_and_ignores_workspace(algo, dv):
    """sse_backward through the C ABI: every gradient inside canary guards,
    the workspace filled with 0xFF bytes (the chunked form's d = 64 operand
    tiles leave half of each tile unwritten: it must never be read), and the
    results bit-identical to a call on a zero-filled workspace."""
    from sparse_state_linear_router_gb300 import binding
    w = H_.workload_variant("layer_bf16", num_heads=2, num_partitions=4, value_dim=dv)
    inp = synth.make_forward_inputs(w, seed=9, lengths=[300, 1, 0, 260], with_init=True)
    T, S, H = inp.total_tokens, inp.num_seqs, w.num_heads
    c, N, P = w.key_dim, w.num_partitions, w.num_slots
    rng = np.random.default_rng(4)
    cfg = H_.config_of(w, algo)
    t = {n: binding.to_device(getattr(inp, n)) for n in ("q", "k", "v", "g", "logits")}
    cu = torch.from_numpy(inp.cu_seqlens.astype(np.int32)).cuda()
    init = torch.from_numpy(inp.init_state).cuda()
    d_out = binding.to_device(synth.f32_to_bf16_bits(rng.normal(size=(T, H, dv)).astype(np.float32)))
    d_fin = torch.from_numpy((rng.normal(size=(S, H, P, c, dv)) * 0.5).astype(np.float32)).cuda()
    nbytes = binding.sse_backward_workspace_size(cfg, T, S)
    ref = binding.backward(cfg, t["q"], t["k"], t["v"], t["g"], t["logits"], cu, d_out, initial_state=init,
                           d_final_state=d_fin, workspace=torch.zeros(nbytes, dtype=torch.uint8, device="cuda"))
    shapes = {"dq": ((T, H, c), torch.bfloat16), "dk": ((T, H, c), torch.bfloat16),
              "dv": ((T, H, dv), torch.bfloat16), "dg": ((T, H, c), torch.bfloat16),
              "dlogits": ((T, H, N), torch.bfloat16), "d_initial_state": ((S, H, P, c, dv), torch.float32)}
    g = {n: _guarded(*shapes[n]) for n in shapes}
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")
    p = binding._ptr
    st = binding.sse_backward(cfg, p(t["q"]), p(t["k"]), p(t["v"]), p(t["g"]), p(t["logits"]), None, None, p(cu), S,
                              T, p(init), p(d_out), p(d_fin), p(g["dq"][0]), p(g["dk"][0]), p(g["dv"][0]),
                              p(g["dg"][0]), p(g["dlogits"][0]), None, None, p(g["d_initial_state"][0]), p(ws),
                              nbytes, binding._stream())
    torch.cuda.synchronize()
    assert st == binding.SSE_OK
    bad = [n for n, (view, raw) in g.items() if not torch.equal(view, ref[n])]
    nonfinite = {n: int((~torch.isfinite(view.float())).sum()) for n, (view, raw) in g.items()}
    for n, (view, raw) in g.items():
        assert _canaries_intact(raw, view.numel() * view.element_size()), n
    assert not bad, (bad, nonfinite)
