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


def _noalloc(lib, cfg, logits, cu, S, T):
    from sparse_state_linear_router_gb300 import binding
    H, k, N = cfg.num_heads, cfg.top_k, cfg.num_partitions
    idx = torch.full((T, H, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, H, k), -7.0, dtype=torch.float32, device="cuda")
    seg_off = torch.full((S * H * N + 1,), -7, dtype=torch.int32, device="cuda")
    perm = torch.full((H * k * T,), -7, dtype=torch.int32, device="cuda")
    st = lib.sse_route_noalloc(ctypes.byref(cfg), logits.data_ptr(), cu.data_ptr(), S, T, idx.data_ptr(),
                               w.data_ptr(), seg_off.data_ptr(), perm.data_ptr(), binding._stream())
    assert st == binding.SSE_OK, binding.sse_status_string(st)
    return idx, w, seg_off, perm


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


def test_noalloc_route_rejects_sizes_beyond_its_scratch(lib):
    from sparse_state_linear_router_gb300 import binding
    cfg = binding.make_config(16, 128, 128, 64, 2)
    fake = 1 << 20  # never dereferenced: the size check comes first
    T = 1 << 20     # 16 * 64 * (4096 + 2) int32 entries > 4 MiB
    st = lib.sse_route_noalloc(ctypes.byref(cfg), fake, fake, 1, T, fake, None, fake, fake, None)
    assert st == binding.SSE_ERR_WORKSPACE
