"""sse_route_noalloc: the routing entry point for callers that cannot
allocate device memory (for example a plugin whose host application owns all
device allocations, or a loop that must not pay cudaMalloc's device-wide
synchronisation).  Its scratch is a fixed array inside the library, so the
test checks, through the C ABI, that two calls in a row (the second one
finding the first one's leftovers in that array) give the same routing and
grouping as sse_route with a caller-provided workspace.  Collected last so a
failure here never hides the other tests."""
import ctypes

import numpy as np
import pytest

from sparse_state_linear_router_gb300 import inputs as synth
from tests import _helpers as H_

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_state_linear_router_gb300 import binding
    return binding.load()


def _noalloc(lib, cfg, logits, cu, S, T, with_w=True, group=True):
    from sparse_state_linear_router_gb300 import binding
    H, k, N = cfg.num_heads, cfg.top_k, cfg.num_partitions
    idx = torch.full((T, H, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, H, k), -7.0, dtype=torch.float32, device="cuda") if with_w else None
    seg_off = torch.full((S * H * N + 1,), -7, dtype=torch.int32, device="cuda") if group else None
    perm = torch.full((max(1, H * k * T),), -7, dtype=torch.int32, device="cuda") if group else None
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    st = lib.sse_route_noalloc(ctypes.byref(cfg), ptr(logits), cu.data_ptr(), S, T, idx.data_ptr(),
                               ptr(w), ptr(seg_off), ptr(perm), binding._stream())
    assert st == binding.SSE_OK, binding.sse_status_string(st)
    return idx, w, seg_off, None if perm is None else perm[:H * k * T]


def test_noalloc_route_matches_route_on_two_calls(lib):
    from sparse_state_linear_router_gb300 import binding
    cases = [
        (H_.workload_variant("varlen_bf16", num_heads=4), [700, 0, 129, 1500], 21),
        (H_.workload_variant("small_bf16", num_heads=3, num_partitions=16, top_k=3), [257, 31], 22),
    ]
    for w, lengths, seed in cases:
        inp = synth.make_forward_inputs(w, seed=seed, lengths=lengths)
        cfg = H_.config_of(w)
        logits = binding.to_device(inp.logits)
        cu = torch.from_numpy(inp.cu_seqlens).cuda()
        S, T = inp.num_seqs, inp.total_tokens
        ref = binding.route(cfg, logits, cu)
        idx, wts, seg_off, perm = _noalloc(lib, cfg, logits, cu, S, T)
        torch.cuda.synchronize()
        assert torch.equal(idx, ref["topk_idx"])
        assert torch.equal(seg_off, ref["seg_off"])
        assert torch.equal(perm, ref["perm"])
        np.testing.assert_allclose(wts.cpu().numpy(), ref["topk_w"].cpu().numpy(), rtol=2e-6, atol=1e-7)


def test_noalloc_route_optional_outputs(lib):
    """The documented variants through the no-allocation entry point: no
    router weights (topk_w NULL), routing only without the grouping
    (seg_off = perm = NULL), and an empty batch (num_seqs = 0) -- each
    compared with sse_route the same way."""
    from sparse_state_linear_router_gb300 import binding
    w = H_.workload_variant("small_bf16", num_heads=3, num_partitions=8, top_k=2)
    inp = synth.make_forward_inputs(w, seed=23, lengths=[411, 0, 97])
    cfg = H_.config_of(w)
    logits = binding.to_device(inp.logits)
    cu = torch.from_numpy(inp.cu_seqlens).cuda()
    S, T = inp.num_seqs, inp.total_tokens
    ref = binding.route(cfg, logits, cu)
    idx, wts, seg_off, perm = _noalloc(lib, cfg, logits, cu, S, T, with_w=False)
    idx2, wts2, seg2, perm2 = _noalloc(lib, cfg, logits, cu, S, T, group=False)
    torch.cuda.synchronize()
    assert wts is None and seg2 is None and perm2 is None
    assert torch.equal(idx, ref["topk_idx"]) and torch.equal(idx2, ref["topk_idx"])
    assert torch.equal(seg_off, ref["seg_off"]) and torch.equal(perm, ref["perm"])
    np.testing.assert_allclose(wts2.cpu().numpy(), ref["topk_w"].cpu().numpy(), rtol=2e-6, atol=1e-7)
    # empty batch: nothing launched, outputs untouched
    empty_cu = torch.zeros(1, dtype=torch.int32, device="cuda")
    sentinel = torch.full((1, 3, 2), -7, dtype=torch.int32, device="cuda")
    st = lib.sse_route_noalloc(ctypes.byref(cfg), None, empty_cu.data_ptr(), 0, 0, sentinel.data_ptr(),
                               None, None, None, binding._stream())
    assert st == binding.SSE_OK
    torch.cuda.synchronize()
    assert bool((sentinel == -7).all())


def test_noalloc_route_rejects_sizes_beyond_its_scratch(lib):
    from sparse_state_linear_router_gb300 import binding
    cfg = binding.make_config(16, 128, 128, 64, 2)
    fake = 1 << 20  # never dereferenced: the size check comes first
    T = 1 << 20     # 16 * 64 * (4096 + 2) int32 entries > 4 MiB
    st = lib.sse_route_noalloc(ctypes.byref(cfg), fake, fake, 1, T, fake, None, fake, fake, None)
    assert st == binding.SSE_ERR_WORKSPACE
