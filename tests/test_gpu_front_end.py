"""GPU parity of sse_front_end (tcgen05 GEMM with fused per-block epilogues)
against the float64 front-end oracle, on the same seeded bf16 inputs, through
the C ABI (marked gpu).  Tolerance: max-abs-rel 2e-2 per output tensor (bf16
inputs and outputs, fp32 accumulation over D)."""
import dataclasses

import numpy as np
import pytest

from oracle import front_end as fe_oracle
from sparse_state_linear_router_gb300 import inputs as synth
from tests import _helpers as H_

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

OUTS = ("q", "k", "v", "log_gate", "logits", "q_shared", "k_shared")
ORACLE_KEY = {"log_gate": "g"}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_state_linear_router_gb300 import binding
    binding.load()


def _cfg(w):
    from sparse_state_linear_router_gb300 import binding
    return binding.make_config(w.num_heads, w.key_dim, w.value_dim, w.num_partitions, 2, 1, 1.0, "bf16")


def _run_gpu(w, inp, lora=True, gate_inv_tau=1.0 / 16):
    from sparse_state_linear_router_gb300 import binding
    dv = lambda a: None if a is None else binding.to_device(a)  # noqa: E731
    res = binding.front_end(_cfg(w), dv(inp.x), dv(inp.w_q), dv(inp.w_k), dv(inp.w_v), dv(inp.w_g), dv(inp.w_e),
                            a_q=dv(inp.a_q) if lora else None, b_q=dv(inp.b_q) if lora else None,
                            a_k=dv(inp.a_k) if lora else None, b_k=dv(inp.b_k) if lora else None,
                            gate_inv_tau=gate_inv_tau)
    torch.cuda.synchronize()
    st, flags = binding.sse_read_device_status(res["workspace"].data_ptr(), binding._stream())
    out = {n: (None if res[n] is None else H_.to_numpy(res[n])) for n in OUTS}
    out["flags"] = flags
    return out


def _run_oracle(w, inp, rows=None, lora=True, gate_inv_tau=1.0 / 16):
    x = inp.x if rows is None else inp.x[rows]
    return fe_oracle.front_end(x, inp.w_q, inp.w_k, inp.w_v, inp.w_g, inp.w_e, num_heads=w.num_heads,
                               gate_inv_tau=gate_inv_tau, a_q=inp.a_q if lora else None,
                               b_q=inp.b_q if lora else None, a_k=inp.a_k if lora else None,
                               b_k=inp.b_k if lora else None)


def _compare(gpu, ref, rows=None, lora=True):
    for n in OUTS:
        r = ref[ORACLE_KEY.get(n, n)]
        if not lora and n in ("q_shared", "k_shared"):
            assert gpu[n] is None and r is None
            continue
        g = gpu[n] if rows is None else gpu[n][rows]
        err = H_.max_abs_rel(g, r)
        assert err < H_.TOL_BF16, (n, err)
    assert gpu["flags"] == 0


VARIANTS = {
    # ragged T (2 full tiles + 44 rows), c = d = 64, H*N = 32
    "small_lora": ("front_end_small", {}, True),
    "small_no_lora": ("front_end_small", {}, False),
    # c = d = 128 blocks, H*N = 16 router columns, three K steps
    "c128_lora": ("front_end_small", {"tokens": 257, "hidden": 192, "num_heads": 2, "key_dim": 128,
                                      "value_dim": 128}, True),
    # mixed widths: c = 128, d = 64, H*N = 256 router columns (the widest block)
    "c128_d64_wide_router": ("front_end_small", {"tokens": 384, "hidden": 128, "num_heads": 16, "key_dim": 128,
                                                 "value_dim": 64, "num_partitions": 16}, True),
    # one K step (the LoRA steps then precede the next tile's only step) and
    # about seven tiles per CTA, so every [q | k] tile but the last of a CTA
    # takes the deferred path
    "d64_many_tiles": ("front_end_small", {"tokens": 4096, "hidden": 64, "num_heads": 16, "key_dim": 128,
                                           "value_dim": 128, "num_partitions": 8}, True),
}


@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_front_end_matches_oracle(name):
    wname, over, lora = VARIANTS[name]
    w = dataclasses.replace(synth.FRONT_END_WORKLOADS[wname], **over)
    inp = synth.make_front_end_inputs(w, seed=3)
    gpu = _run_gpu(w, inp, lora=lora)
    _compare(gpu, _run_oracle(w, inp, lora=lora), lora=lora)


def test_front_end_gate_scale():
    """The log-gate scale is the caller's 1/tau: tau = 1 gives logsigmoid itself."""
    w = synth.FRONT_END_WORKLOADS["front_end_small"]
    inp = synth.make_front_end_inputs(w, seed=4)
    gpu = _run_gpu(w, inp, gate_inv_tau=1.0)
    ref = _run_oracle(w, inp, gate_inv_tau=1.0)
    assert H_.max_abs_rel(gpu["log_gate"], ref["g"]) < H_.TOL_BF16
    assert np.all(gpu["log_gate"] <= 0)


def test_front_end_full_size_sampled_rows():
    """The 32768-token, D = 2048 front end in the bench's launch
    configuration; the oracle recomputes 96 sampled tokens (rows are
    independent), spread over the first, middle and last row tiles."""
    w = synth.FRONT_END_WORKLOADS["front_end_bf16"]
    inp = synth.make_front_end_inputs(w, seed=0)
    gpu = _run_gpu(w, inp)
    rng = np.random.default_rng(1)
    T = w.tokens
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(T - 8, T), rng.integers(0, T, 80)]))
    _compare(gpu, _run_oracle(w, inp, rows=rows), rows=rows)


def test_front_end_feeds_forward():
    """Front end then forward on the GPU equals the oracle's front end then the
    oracle's forward (the k rows are softmax-normalised keys, the g rows
    log-gates, as the forward expects)."""
    from sparse_state_linear_router_gb300 import binding
    w = dataclasses.replace(synth.FRONT_END_WORKLOADS["front_end_small"], tokens=640, num_heads=2)
    inp = synth.make_front_end_inputs(w, seed=6)
    dv = binding.to_device
    fe = binding.front_end(_cfg(w), dv(inp.x), dv(inp.w_q), dv(inp.w_k), dv(inp.w_v), dv(inp.w_g), dv(inp.w_e),
                           a_q=dv(inp.a_q), b_q=dv(inp.b_q), a_k=dv(inp.a_k), b_k=dv(inp.b_k))
    cu_np = np.array([0, 250, 251, 640], dtype=np.int32)
    cu = torch.from_numpy(cu_np).cuda()
    cfg = binding.make_config(w.num_heads, w.key_dim, w.value_dim, w.num_partitions, 2, 1, 1.0, "bf16")
    res = binding.forward(cfg, fe["q"], fe["k"], fe["v"], fe["log_gate"], fe["logits"], cu,
                          q_shared=fe["q_shared"], k_shared=fe["k_shared"])
    torch.cuda.synchronize()
    # the oracle's forward on the GPU front end's bf16 outputs (the routing
    # decisions then agree exactly), and the GPU front end against its oracle
    import oracle
    bits = {n: fe[n].cpu().view(torch.int16).numpy().view(np.uint16) for n in OUTS}
    ref = oracle.forward(bits["q"], bits["k"], bits["v"], bits["log_gate"], bits["logits"], cu_np, top_k=2,
                         use_shared=1, q_shared=bits["q_shared"], k_shared=bits["k_shared"])
    assert H_.max_abs_rel(H_.to_numpy(res["out"]), ref["out"]) < H_.TOL_BF16
    assert H_.max_abs_rel(H_.to_numpy(res["final_state"]), ref["final_state"]) < H_.TOL_BF16
    fe_ref = _run_oracle(w, inp)
    assert H_.max_abs_rel(H_.to_numpy(fe["k"]), fe_ref["k"]) < H_.TOL_BF16
