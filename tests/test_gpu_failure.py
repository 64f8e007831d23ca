"""Failure detection of the tensor-core forwards and backward, exercised
without a GPU fault (marked gpu).

The checked build (libsse_checked.so: fwd_chunked.cu, delta_chunked.cu and
backward_chunked.cu with -DSSE_FAULT_INJECT) gives every bounded wait of
those kernels a 50 ms limit and has a switch per kernel: CTA 0's transform
warps withhold one barrier arrival ("Qt / Kt written" of its first chunk), or
CTA 0 of the delta-rule kernel or of the backward's gradient kernel issues
neither its first product round nor its commit.
The waits then run out; the kernel stops, frees its tensor memory and
returns; the host reads SSE_ERR_DEVICE_TIMEOUT.  The next call on the same
workspace and stream, with the switch off, must be correct.  Nothing traps,
faults or waits without a limit."""
import ctypes
import os

import numpy as np
import pytest

from sparse_state_linear_router_gb300 import inputs as synth
from tests import _helpers as H_

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def checked():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_state_linear_router_gb300 import binding, build
    if not os.path.exists(build.LIB_CHECKED):
        build.build()
    lib = ctypes.CDLL(build.LIB_CHECKED)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    cfgp = ctypes.POINTER(binding.sse_config_t)
    lib.sse_forward_workspace_size.restype = sz
    lib.sse_forward_workspace_size.argtypes = [cfgp, i64, i32]
    lib.sse_forward.restype = ctypes.c_int
    lib.sse_forward.argtypes = [cfgp, P, P, P, P, P, P, P, P, i32, i64, P, P, P, P, P, P, sz, P]
    lib.sse_read_device_status.restype = ctypes.c_int
    lib.sse_read_device_status.argtypes = [P, ctypes.POINTER(i32), P]
    lib.sse_get_last_device_error.restype = ctypes.c_int
    lib.sse_get_last_device_error.argtypes = [P, P]
    lib.sse_debug_set_fault.restype = ctypes.c_int
    lib.sse_debug_set_fault.argtypes = [ctypes.c_int]
    lib.sse_debug_set_delta_fault.restype = ctypes.c_int
    lib.sse_debug_set_delta_fault.argtypes = [ctypes.c_int]
    lib.sse_delta_forward_workspace_size.restype = sz
    lib.sse_delta_forward_workspace_size.argtypes = [cfgp, i64, i32]
    lib.sse_delta_forward.restype = ctypes.c_int
    lib.sse_delta_forward.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, i32, i64, P, P, P, P, P, P, sz, P]
    lib.sse_debug_set_bwd_fault.restype = ctypes.c_int
    lib.sse_debug_set_bwd_fault.argtypes = [ctypes.c_int]
    lib.sse_backward_workspace_size.restype = sz
    lib.sse_backward_workspace_size.argtypes = [cfgp, i64, i32]
    lib.sse_backward.restype = ctypes.c_int
    lib.sse_backward.argtypes = [cfgp, P, P, P, P, P, P, P, P, i32, i64, P, P, P, P, P, P, P, P, P, P, P, P, sz, P]
    yield lib
    lib.sse_debug_set_fault(0)
    lib.sse_debug_set_delta_fault(0)
    lib.sse_debug_set_bwd_fault(0)


def test_timeout_is_reported_and_the_next_call_is_correct(checked):
    import oracle
    from sparse_state_linear_router_gb300 import binding
    w = H_.workload_variant("layer_bf16", num_heads=2, num_partitions=4, top_k=2)
    inp = synth.make_forward_inputs(w, seed=9, lengths=[300, 129, 77], with_init=True)
    cfg = H_.config_of(w, "chunked")
    T, S, H = inp.total_tokens, inp.num_seqs, w.num_heads
    t = {n: binding.to_device(getattr(inp, n)) for n in ("q", "k", "v", "g", "logits")}
    cu = torch.from_numpy(inp.cu_seqlens).cuda()
    init = torch.from_numpy(inp.init_state).cuda()
    out = torch.empty((T, H, w.value_dim), dtype=torch.bfloat16, device="cuda")
    fin = torch.empty((S, H, w.num_slots, w.key_dim, w.value_dim), dtype=torch.float32, device="cuda")
    nbytes = checked.sse_forward_workspace_size(ctypes.byref(cfg), T, S)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = binding._stream()

    def call():
        st = checked.sse_forward(ctypes.byref(cfg), t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(),
                                 t["g"].data_ptr(), t["logits"].data_ptr(), None, None, cu.data_ptr(), S, T,
                                 init.data_ptr(), fin.data_ptr(), out.data_ptr(), None, None, ws.data_ptr(), nbytes,
                                 stream)
        assert st == binding.SSE_OK
        flags = ctypes.c_int32(0)
        status = checked.sse_read_device_status(ws.data_ptr(), ctypes.byref(flags), stream)
        return status, flags.value

    assert checked.sse_debug_set_fault(1) == 0
    status, flags = call()          # returns: the kernel gave up its waits and exited
    assert status == binding.SSE_ERR_DEVICE_TIMEOUT, (status, flags)
    assert flags & binding.SSE_DEVICE_TIMEOUT
    assert checked.sse_get_last_device_error(ws.data_ptr(), stream) == binding.SSE_ERR_DEVICE_TIMEOUT

    assert checked.sse_debug_set_fault(0) == 0
    status, flags = call()          # same workspace and stream, no fault
    assert status == binding.SSE_OK and flags == 0, (status, flags)
    ref = oracle.forward(inp.q, inp.k, inp.v, inp.g, inp.logits, inp.cu_seqlens, top_k=w.top_k,
                         use_shared=w.use_shared, initial_state=inp.init_state)
    assert H_.max_abs_rel(H_.to_numpy(out), ref["out"]) < H_.TOL_BF16
    assert H_.max_abs_rel(H_.to_numpy(fin), ref["final_state"]) < H_.TOL_BF16
    assert np.all(np.isfinite(H_.to_numpy(out)))


def test_delta_timeout_is_reported_and_the_next_call_is_correct(checked):
    from oracle import delta as dl
    from sparse_state_linear_router_gb300 import binding
    w = H_.workload_variant("layer_bf16", num_heads=2, num_partitions=4, top_k=2)
    inp = synth.make_delta_inputs(w, seed=11, lengths=[300, 129, 77], with_init=True)
    cfg = H_.config_of(w)  # the chunked form (bf16, c = d = 128)
    T, S, H = inp.total_tokens, inp.num_seqs, w.num_heads
    t = {n: binding.to_device(getattr(inp, n)) for n in ("q", "k", "v", "log_alpha", "beta", "logits")}
    cu = torch.from_numpy(inp.cu_seqlens).cuda()
    init = torch.from_numpy(inp.init_state).cuda()
    out = torch.empty((T, H, w.value_dim), dtype=torch.bfloat16, device="cuda")
    fin = torch.empty((S, H, w.num_slots, w.key_dim, w.value_dim), dtype=torch.float32, device="cuda")
    nbytes = checked.sse_delta_forward_workspace_size(ctypes.byref(cfg), T, S)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = binding._stream()

    def call():
        st = checked.sse_delta_forward(ctypes.byref(cfg), t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(),
                                       t["log_alpha"].data_ptr(), t["beta"].data_ptr(), t["logits"].data_ptr(),
                                       None, None, cu.data_ptr(), S, T, init.data_ptr(), fin.data_ptr(),
                                       out.data_ptr(), None, None, ws.data_ptr(), nbytes, stream)
        assert st == binding.SSE_OK
        flags = ctypes.c_int32(0)
        status = checked.sse_read_device_status(ws.data_ptr(), ctypes.byref(flags), stream)
        return status, flags.value

    assert checked.sse_debug_set_delta_fault(1) == 0
    status, flags = call()          # returns: CTA 0 gave up its wait and exited
    assert status == binding.SSE_ERR_DEVICE_TIMEOUT, (status, flags)
    assert flags & binding.SSE_DEVICE_TIMEOUT

    assert checked.sse_debug_set_delta_fault(0) == 0
    status, flags = call()          # same workspace and stream, no fault
    assert status == binding.SSE_OK and flags == 0, (status, flags)
    ref = dl.delta_forward(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.logits, inp.cu_seqlens,
                           top_k=w.top_k, use_shared=w.use_shared, scale=1.0, initial_state=inp.init_state)
    assert H_.max_abs_rel(H_.to_numpy(out), ref["out"]) < H_.TOL_BF16
    assert H_.max_abs_rel(H_.to_numpy(fin), ref["final_state"]) < H_.TOL_BF16


def test_backward_timeout_is_reported_and_the_next_call_is_correct(checked):
    from oracle import backward as bw
    from sparse_state_linear_router_gb300 import binding
    w = H_.workload_variant("layer_bf16", num_heads=2, num_partitions=4, top_k=2)
    inp = synth.make_forward_inputs(w, seed=12, lengths=[300, 129, 77], with_init=True)
    cfg = H_.config_of(w)  # the chunked backward (bf16, c = d = 128)
    T, S, H, c, d, N = inp.total_tokens, inp.num_seqs, w.num_heads, w.key_dim, w.value_dim, w.num_partitions
    rng = np.random.default_rng(13)
    d_out = synth.f32_to_bf16_bits(rng.normal(size=(T, H, d)).astype(np.float32))
    d_fin = (rng.normal(size=(S, H, w.num_slots, c, d)) * 0.5).astype(np.float32)
    t = {n: binding.to_device(getattr(inp, n)) for n in ("q", "k", "v", "g", "logits")}
    cu = torch.from_numpy(inp.cu_seqlens).cuda()
    init = torch.from_numpy(inp.init_state).cuda()
    dout_t, dfin_t = binding.to_device(d_out), torch.from_numpy(d_fin).cuda()
    e = lambda n: torch.empty((T, H, n), dtype=torch.bfloat16, device="cuda")  # noqa: E731
    g = {"dq": e(c), "dk": e(c), "dv": e(d), "dg": e(c), "dlogits": e(N),
         "d_initial_state": torch.empty((S, H, w.num_slots, c, d), dtype=torch.float32, device="cuda")}
    nbytes = checked.sse_backward_workspace_size(ctypes.byref(cfg), T, S)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = binding._stream()

    def call():
        st = checked.sse_backward(ctypes.byref(cfg), t["q"].data_ptr(), t["k"].data_ptr(), t["v"].data_ptr(),
                                  t["g"].data_ptr(), t["logits"].data_ptr(), None, None, cu.data_ptr(), S, T,
                                  init.data_ptr(), dout_t.data_ptr(), dfin_t.data_ptr(), g["dq"].data_ptr(),
                                  g["dk"].data_ptr(), g["dv"].data_ptr(), g["dg"].data_ptr(), g["dlogits"].data_ptr(),
                                  None, None, g["d_initial_state"].data_ptr(), ws.data_ptr(), nbytes, stream)
        assert st == binding.SSE_OK
        flags = ctypes.c_int32(0)
        status = checked.sse_read_device_status(ws.data_ptr(), ctypes.byref(flags), stream)
        return status, flags.value

    assert checked.sse_debug_set_bwd_fault(1) == 0
    status, flags = call()          # returns: CTA 0 of the gradient kernel gave up its wait and exited
    assert status == binding.SSE_ERR_DEVICE_TIMEOUT, (status, flags)
    assert flags & binding.SSE_DEVICE_TIMEOUT

    assert checked.sse_debug_set_bwd_fault(0) == 0
    status, flags = call()          # same workspace and stream, no fault
    assert status == binding.SSE_OK and flags == 0, (status, flags)
    ref = bw.backward(inp.q, inp.k, inp.v, inp.g, inp.logits, inp.cu_seqlens, d_out, top_k=w.top_k,
                      use_shared=w.use_shared, scale=1.0, initial_state=inp.init_state, d_final_state=d_fin)
    for n in ("dq", "dk", "dv", "dg", "dlogits", "d_initial_state"):
        assert H_.max_abs_rel(H_.to_numpy(g[n]), ref[n]) < H_.TOL_BF16, n
