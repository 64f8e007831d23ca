"""Seeded synthetic workloads for the SSE layer.

This module only draws random tensors and casts them to the storage dtype; it
holds none of the layer's arithmetic (no routing, no recurrence).  Both the
CUDA path (through the binding) and the CPU oracle consume the exact same
stored bits that it produces.

Workload recipe (per tensor, in this draw order, numpy ``default_rng(seed)``):

1. varlen workloads only: ``lengths = integers(lo, hi + 1, num_seqs)``
2. ``q = normal(0, 1, [T, H, c]) / sqrt(c)``
3. ``k = softmax(normal(0, 1, [T, H, c]))`` over the last axis (the caller-side
   key softmax of the SSE layer; the library receives post-softmax keys)
4. ``v = normal(0, 1, [T, H, d])``
5. ``g = logsigmoid(normal(0, 1, [T, H, c])) / 16`` (per-row log forget gate)
6. ``logits = normal(0, sigma_r, [T, H, N])``
7. workloads with a random initial state: ``init = normal(0, init_std, [S, H, P, c, d])``

Every value is computed in float64 and cast to the workload dtype with
round-to-nearest-even (float64 -> float32 -> bfloat16 for bf16 workloads).
Large tensors are drawn in row blocks; numpy's Generator yields the same
stream whether a tensor is drawn in one call or in consecutive blocks.
Decode step ``s`` draws its single-token inputs from seed ``1000 + s``.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "LayerInputs",
    "DecodeInputs",
    "make_forward_inputs",
    "make_decode_inputs",
    "FrontEndWorkload",
    "FRONT_END_WORKLOADS",
    "FrontEndInputs",
    "make_front_end_inputs",
    "make_forward_inputs_device",
    "DeltaInputs",
    "make_delta_inputs",
    "workload_lengths",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                 # "f32" or "bf16" storage of q/k/v/g/logits/out
    num_heads: int
    key_dim: int               # c
    value_dim: int             # d
    num_partitions: int        # N routed partitions
    top_k: int
    use_shared: int            # 1: an always-on shared partition (state slot N)
    sigma_router: float
    lengths: Optional[tuple] = None          # fixed per-sequence lengths
    varlen: Optional[tuple] = None           # (num_seqs, lo, hi) drawn lengths
    init_std: Optional[float] = None         # random initial state std
    decode_batch: Optional[int] = None       # decode workloads: sequences per step
    decode_steps: Optional[int] = None

    @property
    def num_slots(self) -> int:
        return self.num_partitions + self.use_shared


WORKLOADS = {
    # tiny fp32 forward: B=1, T=64, H=1, c=d=16, N=4, k=1, shared
    "tiny_f32": Workload("tiny_f32", "f32", 1, 16, 16, 4, 1, 1, 1.0, lengths=(64,)),
    # bf16 forward: B=2, T=2048, H=4, c=d=64, N=8, k=2, shared
    "small_bf16": Workload("small_bf16", "bf16", 4, 64, 64, 8, 2, 1, 1.0, lengths=(2048,) * 2),
    # 2B-scale layer forward: B=8, T=4096, H=16, c=d=128, N=8, k=2, shared, sigma 1.5
    "layer_bf16": Workload("layer_bf16", "bf16", 16, 128, 128, 8, 2, 1, 1.5, lengths=(4096,) * 8),
    # long-context varlen forward: 16 sequences, L ~ U[1024, 32768], N=16, init ~ N(0, 0.1)
    "varlen_bf16": Workload("varlen_bf16", "bf16", 16, 128, 128, 16, 2, 1, 1.5,
                            varlen=(16, 1024, 32768), init_std=0.1),
    # decode: 256 sequences x H=16, c=d=128, N=16, k=2, shared; 1000 steps
    "decode_bf16": Workload("decode_bf16", "bf16", 16, 128, 128, 16, 2, 1, 1.0,
                            decode_batch=256, decode_steps=1000),
}


# ----------------------------------------------------------------------------
# dtype helpers (storage only)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    rounded = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float32, exact."""
    u = np.ascontiguousarray(u, dtype=np.uint16)
    return (u.astype(np.uint32) << 16).view(np.float32)


def _cast(x64: np.ndarray, dtype: str) -> np.ndarray:
    x32 = x64.astype(np.float32)
    if dtype == "f32":
        return x32
    if dtype == "bf16":
        return f32_to_bf16_bits(x32)
    raise ValueError(dtype)


def _draw(rng, shape, dtype, transform, block_rows=1 << 14):
    """Draw ``normal(0,1,shape)`` row-block by row-block, apply ``transform`` in
    float64 and cast each block to the storage dtype."""
    out_dtype = np.float32 if dtype == "f32" else np.uint16
    out = np.empty(shape, dtype=out_dtype)
    rows = shape[0]
    for r0 in range(0, rows, block_rows):
        r1 = min(rows, r0 + block_rows)
        blk = rng.normal(0.0, 1.0, (r1 - r0,) + tuple(shape[1:]))
        out[r0:r1] = _cast(transform(blk), dtype)
    return out


def _softmax_last(x):
    m = x.max(axis=-1, keepdims=True)
    e = np.exp(x - m)
    return e / e.sum(axis=-1, keepdims=True)


def _logsigmoid(x):
    return -np.logaddexp(0.0, -x)


@dataclasses.dataclass
class LayerInputs:
    """Packed varlen inputs of one forward call (storage dtype arrays)."""
    workload: Workload
    q: np.ndarray            # [T, H, c]
    k: np.ndarray            # [T, H, c]
    v: np.ndarray            # [T, H, d]
    g: np.ndarray            # [T, H, c]   log forget gate
    logits: np.ndarray       # [T, H, N]   router logits
    cu_seqlens: np.ndarray   # [S+1] int32
    init_state: Optional[np.ndarray]  # [S, H, P, c, d] float32 or None

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def num_seqs(self) -> int:
        return len(self.cu_seqlens) - 1


@dataclasses.dataclass
class DecodeInputs:
    workload: Workload
    q: np.ndarray            # [B, H, c]
    k: np.ndarray
    v: np.ndarray            # [B, H, d]
    g: np.ndarray
    logits: np.ndarray       # [B, H, N]


def workload_lengths(w: Workload, seed: int = 0) -> np.ndarray:
    """The sequence lengths make_forward_inputs(w, seed) uses (the first draw
    of a varlen workload's generator)."""
    if w.varlen is not None:
        ns, lo, hi = w.varlen
        return np.random.default_rng(seed).integers(lo, hi + 1, ns)
    return np.asarray(w.lengths, dtype=np.int64)


def make_forward_inputs_device(w: Workload, seed: int = 0, device="cuda", router_bias=None):
    """One forward batch of workload ``w`` drawn on the GPU with torch's
    generator (benchmark inputs at full size in well under a second): the same
    shapes, sequence lengths (workload_lengths) and distributions as
    make_forward_inputs -- q = N(0,1)/sqrt(c), k = softmax over c of N(0,1),
    v = N(0,1), g = logsigmoid(N(0,1))/16, logits = N(0, sigma_r) (+ an
    optional per-partition bias, for load-skew stress runs), initial state
    N(0, init_std) -- but another stream of numbers, so parity tests keep the
    numpy generator.  Returns dict of device tensors (bf16 token tensors, int32
    cu_seqlens, float32 init or None)."""
    import torch
    assert w.dtype == "bf16"
    lengths = workload_lengths(w, seed)
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    T, S = int(cu[-1]), len(lengths)
    H, c, d, N = w.num_heads, w.key_dim, w.value_dim, w.num_partitions
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def normal(*shape):
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)

    out = {
        "q": (normal(T, H, c) / np.sqrt(c)).to(torch.bfloat16),
        "k": torch.softmax(normal(T, H, c), dim=-1).to(torch.bfloat16),
        "v": normal(T, H, d).to(torch.bfloat16),
        "g": (torch.nn.functional.logsigmoid(normal(T, H, c)) / 16.0).to(torch.bfloat16),
    }
    lg = normal(T, H, N) * w.sigma_router
    if router_bias is not None:
        lg = lg + torch.as_tensor(np.asarray(router_bias, dtype=np.float32), device=device)
    out["logits"] = lg.to(torch.bfloat16)
    out["cu_seqlens"] = torch.from_numpy(cu.astype(np.int32)).to(device)
    out["init"] = (normal(S, H, w.num_slots, c, d) * w.init_std) if w.init_std is not None else None
    out["total_tokens"], out["num_seqs"] = T, S
    return out


def make_forward_inputs(w: Workload, seed: int = 0, lengths=None, with_init=None) -> LayerInputs:
    """Generate one forward batch of workload ``w``.

    ``lengths`` overrides the workload's sequence lengths (parity tests at
    reduced sizes); ``with_init`` forces (True) or suppresses (False) a random
    initial state (std ``w.init_std`` or 0.1)."""
    rng = np.random.default_rng(seed)
    if lengths is None:
        if w.varlen is not None:
            ns, lo, hi = w.varlen
            lengths = rng.integers(lo, hi + 1, ns)
        else:
            lengths = w.lengths
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    H, c, d, N = w.num_heads, w.key_dim, w.value_dim, w.num_partitions
    q = _draw(rng, (T, H, c), w.dtype, lambda x: x / np.sqrt(c))
    k = _draw(rng, (T, H, c), w.dtype, _softmax_last)
    v = _draw(rng, (T, H, d), w.dtype, lambda x: x)
    g = _draw(rng, (T, H, c), w.dtype, lambda x: _logsigmoid(x) / 16.0)
    sig = w.sigma_router
    logits = _draw(rng, (T, H, N), w.dtype, lambda x: x * sig)
    init = None
    want_init = (w.init_std is not None) if with_init is None else with_init
    if want_init:
        std = w.init_std if w.init_std is not None else 0.1
        S = len(lengths)
        init = np.empty((S, H, w.num_slots, c, d), dtype=np.float32)
        for s in range(S):
            init[s] = rng.normal(0.0, std, (H, w.num_slots, c, d)).astype(np.float32)
    return LayerInputs(w, q, k, v, g, logits, cu.astype(np.int32), init)


def make_decode_inputs(w: Workload, step: int, batch: Optional[int] = None) -> DecodeInputs:
    """Single-token inputs of decode step ``step`` (seed ``1000 + step``)."""
    rng = np.random.default_rng(1000 + step)
    B = w.decode_batch if batch is None else batch
    H, c, d, N = w.num_heads, w.key_dim, w.value_dim, w.num_partitions
    q = _draw(rng, (B, H, c), w.dtype, lambda x: x / np.sqrt(c))
    k = _draw(rng, (B, H, c), w.dtype, _softmax_last)
    v = _draw(rng, (B, H, d), w.dtype, lambda x: x)
    g = _draw(rng, (B, H, c), w.dtype, lambda x: _logsigmoid(x) / 16.0)
    sig = w.sigma_router
    logits = _draw(rng, (B, H, N), w.dtype, lambda x: x * sig)
    return DecodeInputs(w, q, k, v, g, logits)


# ----------------------------------------------------------------------------
# Front end (projections from the hidden states)
# ----------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class FrontEndWorkload:
    name: str
    tokens: int                # T
    hidden: int                # D
    num_heads: int
    key_dim: int               # c
    value_dim: int             # d
    num_partitions: int        # N
    lora_rank: int             # r of the shared partition's Q/K LoRA (0: none)


FRONT_END_WORKLOADS = {
    # ragged token count (not a multiple of 128), c = d = 64, H x N = 32 router columns
    "front_end_small": FrontEndWorkload("front_end_small", 300, 256, 4, 64, 64, 8, 64),
    # the 2B-scale layer's tokens (8 x 4096) from hidden size 2048: H16, c=d=128, N8, rank-64 LoRA
    "front_end_bf16": FrontEndWorkload("front_end_bf16", 32768, 2048, 16, 128, 128, 8, 64),
}


@dataclasses.dataclass
class FrontEndInputs:
    """Hidden states and projection weights ([out_features, in_features]
    layout), bfloat16 bit patterns."""
    workload: FrontEndWorkload
    x: np.ndarray              # [T, D]
    w_q: np.ndarray            # [H*c, D]
    w_k: np.ndarray            # [H*c, D]
    w_v: np.ndarray            # [H*d, D]
    w_g: np.ndarray            # [H*c, D]
    w_e: np.ndarray            # [H*N, D]
    a_q: Optional[np.ndarray]  # [r, D]
    b_q: Optional[np.ndarray]  # [H*c, r]
    a_k: Optional[np.ndarray]
    b_k: Optional[np.ndarray]


def make_front_end_inputs(w: FrontEndWorkload, seed: int = 0, tokens: Optional[int] = None) -> FrontEndInputs:
    """Recipe (``default_rng(seed)``, this draw order, bf16 storage):
    x = normal(0, 1, [T, D]); w_q, w_k, w_v, w_g = normal(0, 1/sqrt(D));
    w_e = normal(0, 1.5/sqrt(D)) (router logits of std about 1.5);
    LoRA: a_q, a_k = normal(0, 1/sqrt(D), [r, D]), b_q, b_k =
    normal(0, 0.5/sqrt(r), [H*c, r])."""
    rng = np.random.default_rng(seed)
    T = w.tokens if tokens is None else tokens
    D, H, c, d, N, r = w.hidden, w.num_heads, w.key_dim, w.value_dim, w.num_partitions, w.lora_rank
    s = 1.0 / np.sqrt(D)
    x = _draw(rng, (T, D), "bf16", lambda z: z)
    wq = _draw(rng, (H * c, D), "bf16", lambda z: z * s)
    wk = _draw(rng, (H * c, D), "bf16", lambda z: z * s)
    wv = _draw(rng, (H * d, D), "bf16", lambda z: z * s)
    wg = _draw(rng, (H * c, D), "bf16", lambda z: z * s)
    we = _draw(rng, (H * N, D), "bf16", lambda z: z * 1.5 * s)
    aq = bq = ak = bk = None
    if r:
        sb = 0.5 / np.sqrt(r)
        aq = _draw(rng, (r, D), "bf16", lambda z: z * s)
        bq = _draw(rng, (H * c, r), "bf16", lambda z: z * sb)
        ak = _draw(rng, (r, D), "bf16", lambda z: z * s)
        bk = _draw(rng, (H * c, r), "bf16", lambda z: z * sb)
    return FrontEndInputs(w, x, wq, wk, wv, wg, we, aq, bq, ak, bk)


# ----------------------------------------------------------------------------
# SSE on a gated delta-rule transition
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class DeltaInputs:
    """Packed varlen (or single-token decode) inputs of the delta-rule layer."""
    workload: Workload
    q: np.ndarray            # [T, H, c]
    k: np.ndarray            # [T, H, c], unit rows
    v: np.ndarray            # [T, H, d]
    log_alpha: np.ndarray    # [T, H]
    beta: np.ndarray         # [T, H]
    logits: np.ndarray       # [T, H, N]
    cu_seqlens: np.ndarray   # [S+1] int32
    init_state: Optional[np.ndarray]

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def num_seqs(self) -> int:
        return len(self.cu_seqlens) - 1


def _unit_rows(x):
    return x / np.sqrt((x * x).sum(axis=-1, keepdims=True))


def make_delta_inputs(w: Workload, seed: int = 0, lengths=None, with_init=None) -> DeltaInputs:
    """Inputs of the delta-rule layer, numpy ``default_rng(seed)``, in this
    draw order: (varlen) lengths; q = N(0,1)/sqrt(c); k = unit rows of N(0,1)
    (DeltaNet normalises its keys); v = N(0,1); log_alpha = logsigmoid(N(0,1))/16
    and beta = sigmoid(N(0,1)), one per (token, head); logits = N(0, sigma_r);
    initial state N(0, init_std or 0.1).  float64, cast to the workload dtype."""
    rng = np.random.default_rng(seed)
    if lengths is None:
        if w.varlen is not None:
            ns, lo, hi = w.varlen
            lengths = rng.integers(lo, hi + 1, ns)
        else:
            lengths = w.lengths
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    H, c, d, N = w.num_heads, w.key_dim, w.value_dim, w.num_partitions
    q = _draw(rng, (T, H, c), w.dtype, lambda x: x / np.sqrt(c))
    k = _draw(rng, (T, H, c), w.dtype, _unit_rows)
    v = _draw(rng, (T, H, d), w.dtype, lambda x: x)
    la = _draw(rng, (T, H), w.dtype, lambda x: _logsigmoid(x) / 16.0)
    beta = _draw(rng, (T, H), w.dtype, lambda x: 1.0 / (1.0 + np.exp(-x)))
    logits = _draw(rng, (T, H, N), w.dtype, lambda x: x * w.sigma_router)
    init = None
    want_init = (w.init_std is not None) if with_init is None else with_init
    if want_init:
        std = w.init_std if w.init_std is not None else 0.1
        init = rng.normal(0.0, std, (len(lengths), H, w.num_slots, c, d)).astype(np.float32)
    return DeltaInputs(w, q, k, v, la, beta, logits, cu.astype(np.int32), init)
