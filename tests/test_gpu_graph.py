"""The C-ABI calls inside CUDA graphs (marked gpu).

sse_forward and sse_decode_step issue only stream-ordered work on the stream
they are given (no host synchronisation, no allocation: the workspace is the
caller's), so a caller can capture one call into a CUDA graph and replay it
after writing new inputs into the same buffers -- the way to run the
launch-bound small shapes without per-launch host cost.  Each replay must be
bit-identical to a direct call on the same inputs (the path is deterministic:
fixed-order sums, exact integer routing).
"""
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


NAMES = ("q", "k", "v", "g", "logits")


def _capture(fn):
    """Warm up fn on a side stream, then capture one call into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("algo", ["auto", "masked", "recurrent"])
def test_forward_replays_in_a_cuda_graph(algo):
    from sparse_state_linear_router_gb300 import binding
    w = synth.WORKLOADS["small_bf16"]
    lengths = [700, 333, 1]
    cfg = H_.config_of(w, algo)
    sets = [synth.make_forward_inputs(w, seed=s, lengths=lengths, with_init=True) for s in (21, 22)]
    T, S = sets[0].total_tokens, sets[0].num_seqs
    buf = {n: binding.to_device(getattr(sets[0], n)) for n in NAMES}
    cu = torch.from_numpy(sets[0].cu_seqlens.astype(np.int32)).cuda()
    init = torch.from_numpy(sets[0].init_state).cuda()
    out = torch.empty((T, w.num_heads, w.value_dim), dtype=torch.bfloat16, device="cuda")
    fin = torch.empty((S, w.num_heads, w.num_slots, w.key_dim, w.value_dim), dtype=torch.float32, device="cuda")
    ws = binding.forward_workspace(cfg, T, S)

    def call():
        binding.forward(cfg, *(buf[n] for n in NAMES), cu, initial_state=init, out=out, final_state=fin,
                        workspace=ws)

    def load(inp):
        for n in NAMES:
            buf[n].copy_(binding.to_device(getattr(inp, n)))
        init.copy_(torch.from_numpy(inp.init_state))

    refs = []
    for inp in sets:
        load(inp)
        call()
        torch.cuda.synchronize()
        refs.append((out.clone(), fin.clone()))
    g = _capture(call)
    for inp, (o_ref, f_ref) in zip(sets + sets[::-1], refs + refs[::-1]):
        out.zero_()
        fin.zero_()
        load(inp)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, o_ref) and torch.equal(fin, f_ref)


def test_decode_step_replays_in_a_cuda_graph():
    from sparse_state_linear_router_gb300 import binding
    w = synth.WORKLOADS["decode_bf16"]
    B = 16
    cfg = H_.config_of(w)
    toks = [synth.make_decode_inputs(w, s, batch=B) for s in (3, 4, 5)]
    rng = np.random.default_rng(9)
    s0 = torch.from_numpy((rng.normal(size=(B, w.num_heads, w.num_slots, w.key_dim, w.value_dim)) * 0.1)
                          .astype(np.float32)).cuda()
    buf = {n: binding.to_device(getattr(toks[0], n)) for n in NAMES}
    state = s0.clone()
    out = torch.empty((B, w.num_heads, w.value_dim), dtype=torch.bfloat16, device="cuda")

    def call():
        binding.decode_step(cfg, state, *(buf[n] for n in NAMES), out=out)

    # direct: three steps from s0
    outs, states = [], []
    for tok in toks:
        for n in NAMES:
            buf[n].copy_(binding.to_device(getattr(tok, n)))
        call()
        torch.cuda.synchronize()
        outs.append(out.clone())
        states.append(state.clone())
    g = _capture(call)  # the warm-up and capture calls stepped the state: start over
    state.copy_(s0)
    for tok, o_ref, s_ref in zip(toks, outs, states):
        for n in NAMES:
            buf[n].copy_(binding.to_device(getattr(tok, n)))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, o_ref) and torch.equal(state, s_ref)
