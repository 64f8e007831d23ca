"""CPU-only checks of the C ABI: the library builds, loads and exports every
symbol include/sse.h declares; host-side validation rejects bad arguments
before any launch (no GPU needed, no compute call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sparse_state_linear_router_gb300 import binding, build
    build.build()
    return binding.load()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "sse.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sse_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    from sparse_state_linear_router_gb300 import binding
    declared = _declared_functions()
    assert declared, "no declarations parsed"
    assert sorted(binding.EXPORTED) == declared
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    from sparse_state_linear_router_gb300 import binding
    assert binding.sse_abi_version() == 2
    for s in range(7):
        assert binding.sse_status_string(s).startswith("SSE_")
    assert binding.sse_status_string(binding.SSE_ERR_DEVICE_TIMEOUT).startswith("SSE_ERR_DEVICE_TIMEOUT")


def _cfg(**kw):
    from sparse_state_linear_router_gb300 import binding
    base = dict(num_heads=2, key_dim=64, value_dim=64, num_partitions=8, top_k=2, use_shared=1,
                scale=1.0, dtype="bf16", algo="auto")
    base.update(kw)
    return binding.make_config(**base)


FAKE = 1 << 20  # aligned non-null "device" address; never dereferenced


def _fwd(cfg, T=16, S=1, ws=FAKE, ws_bytes=1 << 40, q=FAKE, cu=FAKE, out=FAKE):
    from sparse_state_linear_router_gb300 import binding
    return binding.sse_forward(cfg, q, FAKE, FAKE, FAKE, FAKE, None, None, cu, S, T, None, None,
                               out, None, None, ws, ws_bytes, None)


def test_forward_rejects_bad_arguments(lib):
    from sparse_state_linear_router_gb300 import binding as b
    assert _fwd(_cfg(top_k=0)) == b.SSE_ERR_INVALID_ARG
    assert _fwd(_cfg(top_k=9, num_partitions=8)) == b.SSE_ERR_INVALID_ARG
    assert _fwd(_cfg(num_partitions=65, top_k=2)) == b.SSE_ERR_UNSUPPORTED
    assert _fwd(_cfg(top_k=9, num_partitions=16)) == b.SSE_ERR_UNSUPPORTED
    assert _fwd(_cfg(use_shared=2)) == b.SSE_ERR_INVALID_ARG
    assert _fwd(_cfg(dtype=7)) == b.SSE_ERR_INVALID_ARG
    assert _fwd(_cfg(algo=9)) == b.SSE_ERR_INVALID_ARG
    assert _fwd(_cfg(scale=float("nan"))) == b.SSE_ERR_INVALID_ARG
    assert _fwd(_cfg(key_dim=12)) == b.SSE_ERR_UNSUPPORTED     # 24-byte bf16 rows
    assert _fwd(_cfg(value_dim=100, dtype="f32")) == b.SSE_ERR_UNSUPPORTED
    assert _fwd(_cfg(), q=None) == b.SSE_ERR_INVALID_ARG
    assert _fwd(_cfg(), cu=None) == b.SSE_ERR_INVALID_ARG
    assert _fwd(_cfg(), q=FAKE + 8) == b.SSE_ERR_INVALID_ARG    # misaligned
    assert _fwd(_cfg(), T=-1) == b.SSE_ERR_INVALID_ARG
    assert _fwd(_cfg(), S=0, T=5) == b.SSE_ERR_INVALID_ARG
    assert _fwd(_cfg(), ws=None) == b.SSE_ERR_WORKSPACE
    assert _fwd(_cfg(), ws=FAKE + 128) == b.SSE_ERR_WORKSPACE
    assert _fwd(_cfg(), ws_bytes=64) == b.SSE_ERR_WORKSPACE
    # empty batch: valid, nothing launched
    assert _fwd(_cfg(), S=0, T=0) == b.SSE_OK


def test_decode_and_route_reject_bad_arguments(lib):
    from sparse_state_linear_router_gb300 import binding as b
    cfg = _cfg()
    assert b.sse_decode_step(cfg, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, -1, FAKE, FAKE, None,
                             None, None) == b.SSE_ERR_INVALID_ARG
    assert b.sse_decode_step(cfg, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, 4, None, FAKE, None,
                             None, None) == b.SSE_ERR_INVALID_ARG
    assert b.sse_decode_step(_cfg(value_dim=24, dtype="f32"), FAKE, FAKE, FAKE, FAKE, FAKE, None, None,
                             4, FAKE, FAKE, None, None, None) == b.SSE_ERR_UNSUPPORTED
    # batch 0: valid no-op
    assert b.sse_decode_step(cfg, None, None, None, None, None, None, None, 0, None, None, None,
                             None, None) == b.SSE_OK
    assert b.sse_route(cfg, FAKE, FAKE, 1, 16, None, None, None, None, FAKE, 1 << 30,
                       None) == b.SSE_ERR_INVALID_ARG
    assert b.sse_route(cfg, FAKE, FAKE, 1, 16, FAKE, None, FAKE, None, FAKE, 1 << 30,
                       None) == b.SSE_ERR_INVALID_ARG  # seg_off without perm
    assert b.sse_route(cfg, FAKE, FAKE, 1, 16, FAKE, None, None, None, FAKE, 8,
                       None) == b.SSE_ERR_WORKSPACE


def test_workspace_sizes(lib):
    from sparse_state_linear_router_gb300 import binding as b
    cfg = _cfg()
    small = b.sse_forward_workspace_size(cfg, 100, 2)
    big = b.sse_forward_workspace_size(cfg, 10000, 2)
    assert 0 < small < big and small % 256 == 0
    assert b.sse_forward_workspace_size(_cfg(top_k=0), 100, 2) == 0
    assert b.sse_route_workspace_size(cfg, 100, 2) > 0
    assert b.sse_route_workspace_size(cfg, 0, 1) > 0


def _fe(cfg, D=256, T=300, x=FAKE, a_q=None, qs=None, ws=FAKE, ws_bytes=1 << 40, tau=1.0 / 16):
    from sparse_state_linear_router_gb300 import binding
    lora = a_q is not None
    return binding.sse_front_end(cfg, D, T, x, FAKE, FAKE, FAKE, FAKE, FAKE, a_q, FAKE if lora else None,
                                 FAKE if lora else None, FAKE if lora else None, tau, FAKE, FAKE, FAKE, FAKE,
                                 FAKE, qs, qs, ws, ws_bytes, None)


def test_front_end_rejects_bad_arguments(lib):
    from sparse_state_linear_router_gb300 import binding as b
    cfg = _cfg()
    assert _fe(_cfg(dtype="f32")) == b.SSE_ERR_UNSUPPORTED
    assert _fe(cfg, D=100) == b.SSE_ERR_UNSUPPORTED            # hidden not a multiple of 64
    assert _fe(_cfg(key_dim=96)) == b.SSE_ERR_UNSUPPORTED
    assert _fe(_cfg(num_heads=1, num_partitions=8)) == b.SSE_ERR_UNSUPPORTED  # H*N = 8 columns
    assert _fe(_cfg(num_heads=64, num_partitions=8)) == b.SSE_ERR_UNSUPPORTED  # H*N = 512 columns
    assert _fe(cfg, T=100) == b.SSE_ERR_UNSUPPORTED             # fewer than one 128-token tile
    assert _fe(cfg, T=-1) == b.SSE_ERR_INVALID_ARG
    assert _fe(cfg, tau=float("inf")) == b.SSE_ERR_INVALID_ARG
    assert _fe(cfg, x=None) == b.SSE_ERR_INVALID_ARG
    assert _fe(cfg, x=FAKE + 8) == b.SSE_ERR_INVALID_ARG        # misaligned
    assert _fe(cfg, a_q=FAKE, qs=None) == b.SSE_ERR_INVALID_ARG  # LoRA without shared outputs
    assert _fe(cfg, ws=None) == b.SSE_ERR_WORKSPACE
    assert _fe(cfg, ws=FAKE + 128) == b.SSE_ERR_WORKSPACE
    assert _fe(cfg, ws_bytes=64) == b.SSE_ERR_WORKSPACE
    small = b.sse_front_end_workspace_size(cfg, 256, 300)
    assert small % 256 == 0 and small >= 256 + 300 * 128 * 2
    assert b.sse_front_end_workspace_size(cfg, 256, 3000) > small


def test_nvtx_build_compiles(tmp_path):
    """The optional NVTX ranges (-DSSE_NVTX, SSE_NVTX=1 for build.py) compile."""
    import subprocess
    from sparse_state_linear_router_gb300 import build
    src = os.path.join(build.CSRC, "sse_api.cu")
    r = subprocess.run([build._nvcc(), *build.ARCH, *build.FLAGS, "-DSSE_NVTX", "-c", src, "-o",
                        str(tmp_path / "api.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_size_limits_rejected_before_launch(lib):
    """Sizes past the kernels' 32-bit row and record indices, and the masking
    schedule's sequence-count limit, are refused on the host."""
    from sparse_state_linear_router_gb300 import binding as b
    cfg = _cfg(num_heads=16, num_partitions=8, top_k=2)
    # T * H * k records must fit in 31 bits
    assert _fwd(cfg, T=(1 << 31) // 32 + 1, S=1) == b.SSE_ERR_UNSUPPORTED
    assert b.sse_forward_workspace_size(cfg, (1 << 31) // 32 + 1, 1) == 0
    # the masking schedule's placement kernel holds one entry per sequence in shared memory
    assert _fwd(_cfg(algo="masked"), T=12001, S=12001) == b.SSE_ERR_UNSUPPORTED
    # decode: batch * H must fit in 31 bits
    assert b.sse_decode_step(_cfg(num_heads=64), FAKE, FAKE, FAKE, FAKE, FAKE, None, None, (1 << 31) // 64,
                             FAKE, FAKE, None, None, None) == b.SSE_ERR_UNSUPPORTED


def test_noalloc_route_checks_match_route(lib):
    """sse_route_noalloc runs the same configuration and size checks as
    sse_route: a bad argument gets the same status from both, before any
    launch (the size limit of the no-allocation scratch aside)."""
    from sparse_state_linear_router_gb300 import binding as b
    bad = [
        (_cfg(top_k=0), 1, 16),
        (_cfg(top_k=9, num_partitions=8), 1, 16),
        (_cfg(num_partitions=65, top_k=2), 1, 16),
        (_cfg(top_k=9, num_partitions=16), 1, 16),
        (_cfg(use_shared=2), 1, 16),
        (_cfg(dtype=7), 1, 16),
        (_cfg(algo=9), 1, 16),
        (_cfg(scale=float("inf")), 1, 16),
        (_cfg(key_dim=12), 1, 16),
        (_cfg(num_heads=1 << 17), 1, 16),
        (_cfg(), -1, 16),
        (_cfg(), 1, -1),
        (_cfg(), 0, 5),
        (_cfg(num_heads=16), 1, (1 << 31) // 32 + 1),
        (_cfg(), 1, 1 << 40),    # total_tokens past 2^31: refused before any product is formed
        (_cfg(), 1, (1 << 63) - 1),
    ]
    for cfg, S, T in bad:
        st_route = b.sse_route(cfg, FAKE, FAKE, S, T, FAKE, None, None, None, FAKE, 1 << 40, None)
        st_noalloc = lib.sse_route_noalloc(ctypes.byref(cfg), FAKE, FAKE, S, T, FAKE, None, None, None, None)
        assert st_route != b.SSE_OK
        assert st_noalloc == st_route, (cfg.num_heads, cfg.top_k, S, T, st_noalloc, st_route)
    # argument pointers: same rules
    cfg = _cfg()
    assert lib.sse_route_noalloc(ctypes.byref(cfg), FAKE, FAKE, 1, 16, None, None, None, None,
                                 None) == b.SSE_ERR_INVALID_ARG
    assert lib.sse_route_noalloc(ctypes.byref(cfg), FAKE, FAKE, 1, 16, FAKE, None, FAKE, None,
                                 None) == b.SSE_ERR_INVALID_ARG
    assert lib.sse_route_noalloc(ctypes.byref(cfg), FAKE + 8, FAKE, 1, 16, FAKE, None, None, None,
                                 None) == b.SSE_ERR_INVALID_ARG
    assert lib.sse_route_noalloc(None, FAKE, FAKE, 1, 16, FAKE, None, None, None, None) == b.SSE_ERR_INVALID_ARG
    # an empty batch is valid and launches nothing
    assert lib.sse_route_noalloc(ctypes.byref(cfg), None, FAKE, 0, 0, FAKE, None, None, None, None) == b.SSE_OK


def test_device_status_readers_reject_bad_workspace(lib):
    """sse_read_device_status / sse_get_last_device_error validate the
    workspace pointer on the host (null or not 256-byte aligned) before any
    copy."""
    from sparse_state_linear_router_gb300 import binding as b
    assert b.sse_get_last_device_error(None, None) == b.SSE_ERR_INVALID_ARG
    assert b.sse_get_last_device_error(FAKE + 64, None) == b.SSE_ERR_INVALID_ARG
    assert b.sse_read_device_status(None, None)[0] == b.SSE_ERR_INVALID_ARG


def _bwd(cfg, T=16, S=1, q=FAKE, qs=None, dqs=None, ks=None, dks=None, ws=FAKE, ws_bytes=1 << 40, dq=FAKE):
    from sparse_state_linear_router_gb300 import binding
    return binding.sse_backward(cfg, q, FAKE, FAKE, FAKE, FAKE, qs, ks, FAKE, S, T, None, FAKE, None, dq, FAKE, FAKE,
                                FAKE, FAKE, dqs, dks, None, ws, ws_bytes, None)


def test_backward_rejects_bad_arguments(lib):
    """sse_backward validates on the host before any launch: the shared
    configuration and size checks, required pointers, alignment, the pairing
    of separate shared q / k with their gradient buffers, the workspace."""
    from sparse_state_linear_router_gb300 import binding as b
    assert _bwd(_cfg(top_k=0)) == b.SSE_ERR_INVALID_ARG
    assert _bwd(_cfg(num_partitions=65, top_k=2)) == b.SSE_ERR_UNSUPPORTED
    assert _bwd(_cfg(key_dim=12)) == b.SSE_ERR_UNSUPPORTED
    assert _bwd(_cfg(value_dim=48, dtype="f32")) == b.SSE_ERR_UNSUPPORTED   # no kernel for d = 48
    assert _bwd(_cfg(), q=None) == b.SSE_ERR_INVALID_ARG
    assert _bwd(_cfg(), dq=None) == b.SSE_ERR_INVALID_ARG
    assert _bwd(_cfg(), q=FAKE + 8) == b.SSE_ERR_INVALID_ARG
    assert _bwd(_cfg(), qs=FAKE) == b.SSE_ERR_INVALID_ARG           # q_shared without dq_shared
    assert _bwd(_cfg(), dks=FAKE) == b.SSE_ERR_INVALID_ARG          # dk_shared without k_shared
    assert _bwd(_cfg(), T=-1) == b.SSE_ERR_INVALID_ARG
    assert _bwd(_cfg(), ws=None) == b.SSE_ERR_WORKSPACE
    assert _bwd(_cfg(), ws_bytes=64) == b.SSE_ERR_WORKSPACE
    assert _bwd(_cfg(), S=0, T=0) == b.SSE_OK
    assert b.sse_backward_workspace_size(_cfg(), 100, 2) > b.sse_forward_workspace_size(_cfg(algo="recurrent"), 0, 1)
    assert b.sse_backward_workspace_size(_cfg(top_k=0), 100, 2) == 0
