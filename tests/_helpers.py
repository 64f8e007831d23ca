"""Shared test helpers: error metric, oracle/GPU runners on the same seeded bits."""
from __future__ import annotations

import numpy as np

import oracle
from sparse_state_linear_router_gb300 import inputs as synth

# Tolerances (max-abs-rel, see max_abs_rel): bf16 token tensors with float32
# accumulation, and the float32 path.
TOL_BF16 = 2e-2
TOL_F32 = 1e-4


def max_abs_rel(x, ref) -> float:
    """max |x - ref| / max(max |ref|, 1e-6), per tensor."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    assert np.all(np.isfinite(x)), "non-finite values in the result"
    return float(np.max(np.abs(x - ref)) / max(float(np.max(np.abs(ref))) if ref.size else 0.0, 1e-6))


def tol_for(w: synth.Workload) -> float:
    return TOL_F32 if w.dtype == "f32" else TOL_BF16


def to_numpy(t) -> np.ndarray:
    """torch tensor (bf16 or f32 or int) -> numpy (bf16 upcast exactly to float32)."""
    import torch
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.float().numpy()
    return t.numpy()


def workload_variant(name: str, **kw) -> synth.Workload:
    import dataclasses
    return dataclasses.replace(synth.WORKLOADS[name], **kw)


def config_of(w: synth.Workload, algo="auto", scale=1.0):
    from sparse_state_linear_router_gb300 import binding
    return binding.make_config(w.num_heads, w.key_dim, w.value_dim, w.num_partitions, w.top_k,
                               w.use_shared, scale, w.dtype, algo)


def run_gpu_forward(w: synth.Workload, inp: synth.LayerInputs, algo="auto", scale=1.0,
                    q_shared=None, k_shared=None):
    import torch
    from sparse_state_linear_router_gb300 import binding
    cfg = config_of(w, algo, scale)
    dev = "cuda"
    t = {n: binding.to_device(getattr(inp, n), dev) for n in ("q", "k", "v", "g", "logits")}
    cu = torch.from_numpy(inp.cu_seqlens.astype(np.int32)).to(dev)
    init = None if inp.init_state is None else torch.from_numpy(inp.init_state).to(dev)
    qs = None if q_shared is None else binding.to_device(q_shared, dev)
    ks = None if k_shared is None else binding.to_device(k_shared, dev)
    res = binding.forward(cfg, t["q"], t["k"], t["v"], t["g"], t["logits"], cu, q_shared=qs,
                          k_shared=ks, initial_state=init, want_routing=True)
    torch.cuda.synchronize()
    st, flags = binding.sse_read_device_status(res["workspace"].data_ptr(), binding._stream())
    return {"out": to_numpy(res["out"]), "final_state": to_numpy(res["final_state"]),
            "topk_idx": to_numpy(res["topk_idx"]), "topk_w": to_numpy(res["topk_w"]),
            "device_flags": flags, "device_status": st}


def run_oracle_forward(w: synth.Workload, inp: synth.LayerInputs, scale=1.0, pairs=None,
                       q_shared=None, k_shared=None):
    return oracle.forward(inp.q, inp.k, inp.v, inp.g, inp.logits, inp.cu_seqlens, top_k=w.top_k,
                          use_shared=w.use_shared, scale=scale, q_shared=q_shared,
                          k_shared=k_shared, initial_state=inp.init_state, pairs=pairs)


def pair_rows(inp: synth.LayerInputs, H: int, pairs):
    """(token indices, head) for each (b*H + h) pair."""
    rows = []
    for p in pairs:
        b, h = divmod(int(p), H)
        rows.append((np.arange(inp.cu_seqlens[b], inp.cu_seqlens[b + 1]), h))
    return rows
