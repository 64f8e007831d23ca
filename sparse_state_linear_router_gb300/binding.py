"""Thin ctypes binding of libsse (include/sse.h).

The functions named like the C entry points (``sse_route``, ``sse_forward``,
``sse_decode_step``, ...) take raw integers (device pointers, sizes, a CUDA
stream handle) and only marshal arguments.  The ``route`` / ``forward`` /
``decode_step`` helpers take torch tensors, allocate outputs and the
workspace with torch (device memory plumbing only) and call the C entry
points on the current torch stream.  Every step of the layer runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback: if libsse.so is
missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libsse.so")

(SSE_OK, SSE_ERR_INVALID_ARG, SSE_ERR_UNSUPPORTED, SSE_ERR_WORKSPACE, SSE_ERR_CUDA, SSE_ERR_DEVICE,
 SSE_ERR_DEVICE_TIMEOUT) = range(7)
# device-status bits (sse_read_device_status)
SSE_DEVICE_TIMEOUT, SSE_DEVICE_RECOMPUTED = 2, 4
SSE_F32, SSE_BF16 = 0, 1
SSE_ALGO_AUTO, SSE_ALGO_CHUNKED, SSE_ALGO_RECURRENT, SSE_ALGO_MASKED = 0, 1, 2, 3
_ALGOS = {"auto": SSE_ALGO_AUTO, "chunked": SSE_ALGO_CHUNKED, "recurrent": SSE_ALGO_RECURRENT,
          "masked": SSE_ALGO_MASKED}

# Every extern "C" symbol that include/sse.h declares.
EXPORTED = ("sse_abi_version", "sse_status_string", "sse_route_workspace_size", "sse_route",
            "sse_route_noalloc", "sse_forward_workspace_size", "sse_forward", "sse_forward_timed", "sse_decode_step",
            "sse_front_end_workspace_size", "sse_front_end", "sse_read_device_status",
            "sse_get_last_device_error", "sse_backward_workspace_size", "sse_backward",
            "sse_delta_forward_workspace_size", "sse_delta_forward", "sse_delta_decode_step")


class sse_config_t(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int32), ("key_dim", ctypes.c_int32),
                ("value_dim", ctypes.c_int32), ("num_partitions", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("use_shared", ctypes.c_int32),
                ("scale", ctypes.c_float), ("dtype", ctypes.c_int32), ("algo", ctypes.c_int32)]


class SSEError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {sse_status_string(status)} (status {status})")
        self.status = status


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libsse.so.  Raises when the library has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libsse.so not found at {path}; build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    cfgp = ctypes.POINTER(sse_config_t)
    lib.sse_abi_version.restype = i32
    lib.sse_abi_version.argtypes = []
    lib.sse_status_string.restype = ctypes.c_char_p
    lib.sse_status_string.argtypes = [ctypes.c_int]
    lib.sse_route_workspace_size.restype = sz
    lib.sse_route_workspace_size.argtypes = [cfgp, i64, i32]
    lib.sse_route.restype = ctypes.c_int
    lib.sse_route.argtypes = [cfgp, P, P, i32, i64, P, P, P, P, P, sz, P]
    lib.sse_route_noalloc.restype = ctypes.c_int
    lib.sse_route_noalloc.argtypes = [cfgp, P, P, i32, i64, P, P, P, P, P]
    lib.sse_forward_workspace_size.restype = sz
    lib.sse_forward_workspace_size.argtypes = [cfgp, i64, i32]
    lib.sse_forward.restype = ctypes.c_int
    lib.sse_forward.argtypes = [cfgp, P, P, P, P, P, P, P, P, i32, i64, P, P, P, P, P, P, sz, P]
    lib.sse_forward_timed.restype = ctypes.c_int
    lib.sse_forward_timed.argtypes = [cfgp, P, P, P, P, P, P, P, P, i32, i64, P, P, P, P, P, P, sz, P,
                                      P, ctypes.POINTER(i32)]
    lib.sse_decode_step.restype = ctypes.c_int
    lib.sse_decode_step.argtypes = [cfgp, P, P, P, P, P, P, P, i32, P, P, P, P, P]
    lib.sse_front_end_workspace_size.restype = sz
    lib.sse_front_end_workspace_size.argtypes = [cfgp, i32, i64]
    lib.sse_front_end.restype = ctypes.c_int
    lib.sse_front_end.argtypes = [cfgp, i32, i64, P, P, P, P, P, P, P, P, P, P, ctypes.c_float,
                                  P, P, P, P, P, P, P, P, sz, P]
    lib.sse_read_device_status.restype = ctypes.c_int
    lib.sse_read_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_int32), P]
    lib.sse_get_last_device_error.restype = ctypes.c_int
    lib.sse_get_last_device_error.argtypes = [P, P]
    lib.sse_backward_workspace_size.restype = sz
    lib.sse_backward_workspace_size.argtypes = [cfgp, i64, i32]
    lib.sse_backward.restype = ctypes.c_int
    lib.sse_backward.argtypes = [cfgp, P, P, P, P, P, P, P, P, i32, i64, P, P, P, P, P, P, P, P, P, P, P, P, sz, P]
    lib.sse_delta_forward_workspace_size.restype = sz
    lib.sse_delta_forward_workspace_size.argtypes = [cfgp, i64, i32]
    lib.sse_delta_forward.restype = ctypes.c_int
    lib.sse_delta_forward.argtypes = [cfgp, P, P, P, P, P, P, P, P, P, i32, i64, P, P, P, P, P, P, sz, P]
    lib.sse_delta_decode_step.restype = ctypes.c_int
    lib.sse_delta_decode_step.argtypes = [cfgp, P, P, P, P, P, P, P, P, i32, P, P, P, P, P]
    _lib = lib
    return lib


# ---------------------------------------------------------------------------
# Raw C entry points (integers in, status out)
# ---------------------------------------------------------------------------
def sse_abi_version() -> int:
    return load().sse_abi_version()


def sse_status_string(status: int) -> str:
    return load().sse_status_string(status).decode()


def sse_route_workspace_size(cfg: sse_config_t, total_tokens: int, num_seqs: int) -> int:
    return load().sse_route_workspace_size(ctypes.byref(cfg), total_tokens, num_seqs)


def sse_forward_workspace_size(cfg: sse_config_t, total_tokens: int, num_seqs: int) -> int:
    return load().sse_forward_workspace_size(ctypes.byref(cfg), total_tokens, num_seqs)


def sse_route(cfg, logits, cu_seqlens, num_seqs, total_tokens, topk_idx, topk_w, seg_off, perm,
              workspace, workspace_bytes, stream) -> int:
    return load().sse_route(ctypes.byref(cfg), logits, cu_seqlens, num_seqs, total_tokens, topk_idx,
                            topk_w, seg_off, perm, workspace, workspace_bytes, stream)


def sse_forward(cfg, q, k, v, log_gate, logits, q_shared, k_shared, cu_seqlens, num_seqs,
                total_tokens, initial_state, final_state, out, topk_idx, topk_w, workspace,
                workspace_bytes, stream) -> int:
    return load().sse_forward(ctypes.byref(cfg), q, k, v, log_gate, logits, q_shared, k_shared,
                              cu_seqlens, num_seqs, total_tokens, initial_state, final_state, out,
                              topk_idx, topk_w, workspace, workspace_bytes, stream)


def sse_forward_timed(cfg, q, k, v, log_gate, logits, q_shared, k_shared, cu_seqlens, num_seqs,
                      total_tokens, initial_state, final_state, out, topk_idx, topk_w, workspace,
                      workspace_bytes, stream, stage_events=None):
    """Returns (status, kernels launched).  stage_events: 4 raw cudaEvent_t handles or None."""
    ev = None
    if stage_events is not None:
        ev = (ctypes.c_void_p * 4)(*stage_events)
    n = ctypes.c_int32(0)
    st = load().sse_forward_timed(ctypes.byref(cfg), q, k, v, log_gate, logits, q_shared, k_shared,
                                  cu_seqlens, num_seqs, total_tokens, initial_state, final_state, out,
                                  topk_idx, topk_w, workspace, workspace_bytes, stream, ev,
                                  ctypes.byref(n))
    return st, n.value


def sse_decode_step(cfg, q, k, v, log_gate, logits, q_shared, k_shared, batch, state, out,
                    topk_idx, topk_w, stream) -> int:
    return load().sse_decode_step(ctypes.byref(cfg), q, k, v, log_gate, logits, q_shared, k_shared,
                                  batch, state, out, topk_idx, topk_w, stream)


def sse_front_end_workspace_size(cfg: sse_config_t, hidden: int, total_tokens: int) -> int:
    return int(load().sse_front_end_workspace_size(ctypes.byref(cfg), hidden, total_tokens))


def sse_front_end(cfg, hidden, total_tokens, x, w_q, w_k, w_v, w_g, w_e, a_q, b_q, a_k, b_k,
                  gate_inv_tau, q, k, v, log_gate, logits, q_shared, k_shared, workspace,
                  workspace_bytes, stream) -> int:
    return load().sse_front_end(ctypes.byref(cfg), hidden, total_tokens, x, w_q, w_k, w_v, w_g, w_e,
                                a_q, b_q, a_k, b_k, float(gate_inv_tau), q, k, v, log_gate, logits,
                                q_shared, k_shared, workspace, workspace_bytes, stream)


def sse_read_device_status(workspace, stream):
    flags = ctypes.c_int32(0)
    st = load().sse_read_device_status(workspace, ctypes.byref(flags), stream)
    return st, flags.value


def sse_get_last_device_error(workspace, stream) -> int:
    return load().sse_get_last_device_error(workspace, stream)


def sse_backward_workspace_size(cfg: sse_config_t, total_tokens: int, num_seqs: int) -> int:
    return load().sse_backward_workspace_size(ctypes.byref(cfg), total_tokens, num_seqs)


def sse_backward(cfg, q, k, v, log_gate, logits, q_shared, k_shared, cu_seqlens, num_seqs, total_tokens,
                 initial_state, d_out, d_final_state, dq, dk, dv, d_log_gate, d_logits, dq_shared, dk_shared,
                 d_initial_state, workspace, workspace_bytes, stream) -> int:
    return load().sse_backward(ctypes.byref(cfg), q, k, v, log_gate, logits, q_shared, k_shared, cu_seqlens,
                               num_seqs, total_tokens, initial_state, d_out, d_final_state, dq, dk, dv, d_log_gate,
                               d_logits, dq_shared, dk_shared, d_initial_state, workspace, workspace_bytes, stream)


# ---------------------------------------------------------------------------
# torch-tensor helpers (allocation of outputs/workspace + marshalling)
# ---------------------------------------------------------------------------
def make_config(num_heads, key_dim, value_dim, num_partitions, top_k, use_shared=1, scale=1.0,
                dtype="bf16", algo="auto") -> sse_config_t:
    dt = {"bf16": SSE_BF16, "f32": SSE_F32}[dtype] if isinstance(dtype, str) else dtype
    return sse_config_t(num_heads, key_dim, value_dim, num_partitions, top_k, int(use_shared),
                        float(scale), dt, _ALGOS[algo] if isinstance(algo, str) else int(algo))


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def _check(status: int, what: str):
    if status != SSE_OK:
        raise SSEError(status, what)


def _token_dtype(cfg):
    import torch
    return torch.bfloat16 if cfg.dtype == SSE_BF16 else torch.float32


def route(cfg, logits, cu_seqlens, group: bool = True, workspace=None):
    """Returns dict(topk_idx [T,H,k] int32, topk_w [T,H,k] f32, seg_off, perm)."""
    import torch
    T = logits.shape[0]
    S = cu_seqlens.numel() - 1
    H, k, N = cfg.num_heads, cfg.top_k, cfg.num_partitions
    dev = logits.device
    idx = torch.empty((T, H, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, H, k), dtype=torch.float32, device=dev)
    seg_off = torch.empty(S * H * N + 1, dtype=torch.int32, device=dev) if group else None
    perm = torch.empty(max(1, H * k * T), dtype=torch.int32, device=dev) if group else None
    nbytes = sse_route_workspace_size(cfg, T, S)
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    _check(sse_route(cfg, _ptr(logits), _ptr(cu_seqlens), S, T, _ptr(idx), _ptr(w), _ptr(seg_off),
                     _ptr(perm), _ptr(workspace), workspace.numel(), _stream()), "sse_route")
    return {"topk_idx": idx, "topk_w": w, "seg_off": seg_off,
            "perm": None if perm is None else perm[:H * k * T]}


def forward_workspace(cfg, total_tokens: int, num_seqs: int, device="cuda"):
    import torch
    n = sse_forward_workspace_size(cfg, total_tokens, num_seqs)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def forward(cfg, q, k, v, log_gate, logits, cu_seqlens, *, q_shared=None, k_shared=None,
            initial_state=None, want_final_state=True, out=None, final_state=None,
            want_routing=False, workspace=None):
    """SSE forward on device tensors; returns dict(out, final_state, topk_idx, topk_w)."""
    import torch
    T = q.shape[0]
    S = cu_seqlens.numel() - 1
    H, d, c = cfg.num_heads, cfg.value_dim, cfg.key_dim
    P = cfg.num_partitions + cfg.use_shared
    dev = q.device
    if out is None:
        out = torch.empty((T, H, d), dtype=_token_dtype(cfg), device=dev)
    if final_state is None and want_final_state:
        final_state = torch.empty((S, H, P, c, d), dtype=torch.float32, device=dev)
    idx = w = None
    if want_routing:
        idx = torch.empty((T, H, cfg.top_k), dtype=torch.int32, device=dev)
        w = torch.empty((T, H, cfg.top_k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = forward_workspace(cfg, T, S, dev)
    _check(sse_forward(cfg, _ptr(q), _ptr(k), _ptr(v), _ptr(log_gate), _ptr(logits), _ptr(q_shared),
                       _ptr(k_shared), _ptr(cu_seqlens), S, T, _ptr(initial_state), _ptr(final_state),
                       _ptr(out), _ptr(idx), _ptr(w), _ptr(workspace), workspace.numel(), _stream()),
           "sse_forward")
    return {"out": out, "final_state": final_state, "topk_idx": idx, "topk_w": w,
            "workspace": workspace}


def decode_step(cfg, state, q, k, v, log_gate, logits, *, q_shared=None, k_shared=None, out=None,
                want_routing=False):
    """One decode step; ``state`` [B,H,P,c,d] float32 is updated in place."""
    import torch
    B = q.shape[0]
    H, d = cfg.num_heads, cfg.value_dim
    dev = q.device
    if out is None:
        out = torch.empty((B, H, d), dtype=_token_dtype(cfg), device=dev)
    idx = w = None
    if want_routing:
        idx = torch.empty((B, H, cfg.top_k), dtype=torch.int32, device=dev)
        w = torch.empty((B, H, cfg.top_k), dtype=torch.float32, device=dev)
    _check(sse_decode_step(cfg, _ptr(q), _ptr(k), _ptr(v), _ptr(log_gate), _ptr(logits),
                           _ptr(q_shared), _ptr(k_shared), B, _ptr(state), _ptr(out), _ptr(idx),
                           _ptr(w), _stream()), "sse_decode_step")
    return {"out": out, "topk_idx": idx, "topk_w": w}


def backward(cfg, q, k, v, log_gate, logits, cu_seqlens, d_out, *, q_shared=None, k_shared=None,
             initial_state=None, d_final_state=None, want_d_initial_state=True, workspace=None):
    """Gradients of <d_out, out> + <d_final_state, final_state> on device
    tensors; returns dict(dq, dk, dv, dg, dlogits, dq_shared, dk_shared,
    d_initial_state, workspace)."""
    import torch
    T = q.shape[0]
    S = cu_seqlens.numel() - 1
    H, c, d, N = cfg.num_heads, cfg.key_dim, cfg.value_dim, cfg.num_partitions
    P = N + cfg.use_shared
    dev = q.device
    dt = _token_dtype(cfg)
    e = lambda w: torch.empty((T, H, w), dtype=dt, device=dev)  # noqa: E731
    out = {"dq": e(c), "dk": e(c), "dv": e(d), "dg": e(c), "dlogits": e(N),
           "dq_shared": e(c) if q_shared is not None else None,
           "dk_shared": e(c) if k_shared is not None else None,
           "d_initial_state": (torch.empty((S, H, P, c, d), dtype=torch.float32, device=dev)
                               if want_d_initial_state else None)}
    if workspace is None:
        workspace = torch.empty(max(sse_backward_workspace_size(cfg, T, S), 256), dtype=torch.uint8, device=dev)
    _check(sse_backward(cfg, _ptr(q), _ptr(k), _ptr(v), _ptr(log_gate), _ptr(logits), _ptr(q_shared),
                        _ptr(k_shared), _ptr(cu_seqlens), S, T, _ptr(initial_state), _ptr(d_out),
                        _ptr(d_final_state), _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]),
                        _ptr(out["dlogits"]), _ptr(out["dq_shared"]), _ptr(out["dk_shared"]),
                        _ptr(out["d_initial_state"]), _ptr(workspace), workspace.numel(), _stream()),
           "sse_backward")
    return dict(out, workspace=workspace)


def delta_forward(cfg, q, k, v, log_alpha, beta, logits, cu_seqlens, *, q_shared=None, k_shared=None,
                  initial_state=None, want_final_state=True, want_routing=False, workspace=None):
    """SSE on the gated delta rule (sse_delta_forward) on device tensors;
    returns dict(out, final_state, topk_idx, topk_w, workspace)."""
    import torch
    T = q.shape[0]
    S = cu_seqlens.numel() - 1
    H, d, c = cfg.num_heads, cfg.value_dim, cfg.key_dim
    P = cfg.num_partitions + cfg.use_shared
    dev = q.device
    out = torch.empty((T, H, d), dtype=_token_dtype(cfg), device=dev)
    fin = torch.empty((S, H, P, c, d), dtype=torch.float32, device=dev) if want_final_state else None
    idx = w = None
    if want_routing:
        idx = torch.empty((T, H, cfg.top_k), dtype=torch.int32, device=dev)
        w = torch.empty((T, H, cfg.top_k), dtype=torch.float32, device=dev)
    if workspace is None:
        n = load().sse_delta_forward_workspace_size(ctypes.byref(cfg), T, S)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    _check(load().sse_delta_forward(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                    _ptr(logits), _ptr(q_shared), _ptr(k_shared), _ptr(cu_seqlens), S, T,
                                    _ptr(initial_state), _ptr(fin), _ptr(out), _ptr(idx), _ptr(w), _ptr(workspace),
                                    workspace.numel(), _stream()), "sse_delta_forward")
    return {"out": out, "final_state": fin, "topk_idx": idx, "topk_w": w, "workspace": workspace}


def delta_decode_step(cfg, state, q, k, v, log_alpha, beta, logits, *, q_shared=None, k_shared=None,
                      want_routing=False):
    """One delta-rule decode step; ``state`` [B,H,P,c,d] float32 is updated in place."""
    import torch
    B = q.shape[0]
    H, d = cfg.num_heads, cfg.value_dim
    dev = q.device
    out = torch.empty((B, H, d), dtype=_token_dtype(cfg), device=dev)
    idx = w = None
    if want_routing:
        idx = torch.empty((B, H, cfg.top_k), dtype=torch.int32, device=dev)
        w = torch.empty((B, H, cfg.top_k), dtype=torch.float32, device=dev)
    _check(load().sse_delta_decode_step(ctypes.byref(cfg), _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                        _ptr(logits), _ptr(q_shared), _ptr(k_shared), B, _ptr(state), _ptr(out),
                                        _ptr(idx), _ptr(w), _stream()), "sse_delta_decode_step")
    return {"out": out, "topk_idx": idx, "topk_w": w}


def front_end(cfg, x, w_q, w_k, w_v, w_g, w_e, *, a_q=None, b_q=None, a_k=None, b_k=None,
              gate_inv_tau=1.0 / 16.0, outs=None, workspace=None):
    """Projections from the hidden states x [T, D] (bf16 device tensors);
    returns dict(q, k, v, log_gate, logits, q_shared, k_shared, workspace)."""
    import torch
    T, D = x.shape
    H, c, d, N = cfg.num_heads, cfg.key_dim, cfg.value_dim, cfg.num_partitions
    dev = x.device
    lora = a_q is not None
    if outs is None:
        e = lambda w: torch.empty((T, H, w), dtype=torch.bfloat16, device=dev)  # noqa: E731
        outs = {"q": e(c), "k": e(c), "v": e(d), "log_gate": e(c), "logits": e(N),
                "q_shared": e(c) if lora else None, "k_shared": e(c) if lora else None}
    if workspace is None:
        workspace = torch.empty(max(sse_front_end_workspace_size(cfg, D, T), 256), dtype=torch.uint8,
                                device=dev)
    _check(sse_front_end(cfg, D, T, _ptr(x), _ptr(w_q), _ptr(w_k), _ptr(w_v), _ptr(w_g), _ptr(w_e),
                         _ptr(a_q), _ptr(b_q), _ptr(a_k), _ptr(b_k), gate_inv_tau, _ptr(outs["q"]),
                         _ptr(outs["k"]), _ptr(outs["v"]), _ptr(outs["log_gate"]), _ptr(outs["logits"]),
                         _ptr(outs["q_shared"]), _ptr(outs["k_shared"]), _ptr(workspace), workspace.numel(),
                         _stream()), "sse_front_end")
    return dict(outs, workspace=workspace)


def to_device(arr, device="cuda"):
    """numpy storage array (float32, or bf16 bits in uint16) -> torch tensor."""
    import numpy as np
    import torch
    if arr.dtype == np.uint16:
        return torch.from_numpy(arr.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)
