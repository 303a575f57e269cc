"""Seeded synthetic inputs for the fused input projection.

This module is shared by the CPU oracle's tests and by the GPU path's tests and
benchmark. It holds no arithmetic of the projection itself: it only draws
numbers and lays them out in the shapes of the workloads.

Generator: counter-based. Value ``i`` of stream ``(seed, stream_id)`` is a pure
function of those three integers, so any subset of a tensor can be regenerated
without generating the rest.

* splitmix64 (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) mixes the counter ``key + (i + 1) * golden_gamma``.
* Box-Muller (G. Box, M. Muller, 1958) turns two 53-bit uniforms into one
  standard normal (the cosine branch).

Distributions follow the workloads: activations ~ N(0, 1), weights ~ N(0, 1/C),
bias ~ N(0, 0.02), where the second argument is the variance.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Tuple

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

ACT_NONE, ACT_GELU_ERF, ACT_GELU_TANH, ACT_SILU, ACT_RELU2 = 0, 1, 2, 3, 4
ACT_NAMES = {ACT_NONE: "none", ACT_GELU_ERF: "gelu", ACT_GELU_TANH: "gelu_tanh", ACT_SILU: "silu",
             ACT_RELU2: "relu2"}

# stream ids of the tensors one workload draws
STREAM_X, STREAM_W, STREAM_B = 1, 2, 3
STREAM_GFF, STREAM_GQ, STREAM_GK, STREAM_GV = 4, 5, 6, 7  # upstream gradients (backward)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    s = np.array([(seed & 0xFFFFFFFF) << 32 | (stream & 0xFFFFFFFF)], dtype=np.uint64)
    return _mix(s + _GAMMA)[0]


def uniform53(seed: int, stream: int, start: int, n: int) -> np.ndarray:
    """n uniforms in (0, 1], counters start .. start+n-1."""
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = _mix(_key(seed, stream) + ctr * _GAMMA)
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (1.0 / 9007199254740992.0)


def normal(seed: int, stream: int, n: int, start: int = 0, chunk: int = 1 << 22) -> np.ndarray:
    """n standard normals; element i uses uniforms 2i and 2i+1 of the stream."""
    out = np.empty(n, dtype=np.float64)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        u = uniform53(seed, stream, 2 * (start + lo), 2 * (hi - lo))
        u1, u2 = u[0::2], u[1::2]
        out[lo:hi] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return out


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    bits = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    bias = ((bits >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((bits + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape of one projection problem.

    ``x_shape`` is the activation's logical shape, stored contiguously; axis
    ``channel_dim`` holds C; of the other axes, the first ``n_batch_dims`` form
    the batch index b and the rest (in order) the token index t.
    """
    name: str
    x_shape: Tuple[int, ...]
    channel_dim: int
    n_batch_dims: int
    C: int
    F: int
    heads: int
    head_dim: int
    act: int
    rope_base: float  # <= 0: no rotary embedding
    bias: bool
    dtype: str  # "bf16" | "f32"
    seed: int
    rope_n_elem: int = 0  # 0: the whole head is rotated
    n_query_groups: int = 0  # 0: one k/v head per q head, blocked [q|k|v] columns
    k_transposed: bool = False  # k emitted [B*kv, head_dim, T]

    @property
    def N(self) -> int:
        if self.n_query_groups:
            return self.F + (self.heads + 2 * self.n_query_groups) * self.head_dim
        return self.F + 3 * self.heads * self.head_dim

    @property
    def tokens_axes(self) -> Tuple[int, ...]:
        return tuple(s for a, s in enumerate(self.x_shape) if a != self.channel_dim)

    @property
    def Bb(self) -> int:
        return int(np.prod(self.tokens_axes[: self.n_batch_dims], dtype=np.int64))

    @property
    def T(self) -> int:
        return int(np.prod(self.tokens_axes[self.n_batch_dims:], dtype=np.int64))

    @property
    def M(self) -> int:
        return self.Bb * self.T

    @property
    def flops(self) -> int:
        return 2 * self.M * self.C * self.N

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads of the fused-projection benchmark, named by what they are.
WORKLOADS: Dict[str, Workload] = {
    # tiny channels-first fp32 block: x [1, 32, 8, 8, 1]
    "tiny_fp32": Workload("tiny_fp32", (1, 32, 8, 8, 1), 1, 1, 32, 64, 2, 16,
                          ACT_GELU_TANH, 10000.0, True, "f32", 0),
    # Walrus-shaped processor block: x [B=4, T=6, C=768, 32, 32, 1], 24 576 tokens
    "walrus_bf16": Workload("walrus_bf16", (4, 6, 768, 32, 32, 1), 2, 1, 768, 3072, 12, 64,
                            ACT_GELU_ERF, 10000.0, True, "bf16", 1),
    # BERT-base MLP fused linear: x [16, 512, 768] -> 3072, bias + GELU
    "bert_ff_bf16": Workload("bert_ff_bf16", (16, 512, 768), 2, 1, 768, 3072, 0, 0,
                             ACT_GELU_ERF, 0.0, True, "bf16", 2),
    # BERT-base attention projection wx+b into q, k, v (12 x 64)
    "bert_qkv_bf16": Workload("bert_qkv_bf16", (16, 512, 768), 2, 1, 768, 0, 12, 64,
                              ACT_NONE, 0.0, True, "bf16", 2),
    # LLM QKV split + rotary: x [2, 4096, 4096], 32 x 128, no bias
    "llm_qkv_rope_bf16": Workload("llm_qkv_rope_bf16", (2, 4096, 4096), 2, 1, 4096, 0, 32, 128,
                                  ACT_NONE, 10000.0, False, "bf16", 3),
    # diffusion-UNet attention projection on NCHW x [2, 320, 64, 64], 5 x 64
    "unet_qkv_bf16": Workload("unet_qkv_bf16", (2, 320, 64, 64), 1, 1, 320, 0, 5, 64,
                              ACT_NONE, 0.0, False, "bf16", 4),
    "unet_qkv_fp32": Workload("unet_qkv_fp32", (2, 320, 64, 64), 1, 1, 320, 0, 5, 64,
                              ACT_NONE, 0.0, False, "f32", 4),
    # grouped-query QKV split + partial rotary of the RoPE fusion issue's toy
    # config: x [2, 1024, 512], 16 heads x 32, 4 query groups, 8 rotated lanes
    "gqa_rope_toy_bf16": Workload("gqa_rope_toy_bf16", (2, 1024, 512), 2, 1, 512, 0, 16, 32,
                                  ACT_NONE, 10000.0, False, "bf16", 5, rope_n_elem=8,
                                  n_query_groups=4),
}


def _to_dtype(a64: np.ndarray, dtype: str) -> np.ndarray:
    a32 = a64.astype(np.float32)
    return f32_to_bf16_bits(a32) if dtype == "bf16" else a32


def make_inputs(w: Workload, seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Draw x, W, bias for workload ``w``.

    Returns host arrays: bf16 data as uint16 bits, f32 data as float32. ``x`` has
    shape ``w.x_shape`` (contiguous), ``W`` is [C, N] row-major, ``b`` is [N] or
    None, ``pos`` is None (positions 0..T-1).
    """
    seed = w.seed if seed is None else seed
    nx = int(np.prod(w.x_shape, dtype=np.int64))
    x = _to_dtype(normal(seed, STREAM_X, nx), w.dtype).reshape(w.x_shape)
    W = _to_dtype(normal(seed, STREAM_W, w.C * w.N) * np.sqrt(1.0 / w.C), w.dtype)
    W = W.reshape(w.C, w.N)
    b = _to_dtype(normal(seed, STREAM_B, w.N) * np.sqrt(0.02), w.dtype) if w.bias else None
    return {"x": x, "W": W, "b": b, "pos": None}


def make_grads(w: Workload, seed: Optional[int] = None) -> Dict[str, Optional[np.ndarray]]:
    """Draw upstream gradients for the backward of workload ``w``: N(0, 1)
    values in the forward's output layouts and dtype — ff [M, F], q
    [B*heads, T, hd], k [B*kv, T, hd] (or [B*kv, hd, T] pre-transposed), v
    [B*kv, T, hd]; None for an empty block."""
    seed = w.seed if seed is None else seed
    nkv = w.n_query_groups or w.heads
    B, T, hd = w.Bb, w.T, w.head_dim

    def draw(stream, shape):
        n = int(np.prod(shape, dtype=np.int64))
        return _to_dtype(normal(seed, stream, n), w.dtype).reshape(shape)

    out: Dict[str, Optional[np.ndarray]] = {"ff": None, "q": None, "k": None, "v": None}
    if w.F:
        out["ff"] = draw(STREAM_GFF, (w.M, w.F))
    if w.heads:
        out["q"] = draw(STREAM_GQ, (B * w.heads, T, hd))
        out["k"] = draw(STREAM_GK, (B * nkv, hd, T) if w.k_transposed else (B * nkv, T, hd))
        out["v"] = draw(STREAM_GV, (B * nkv, T, hd))
    return out


def as_float64(a: Optional[np.ndarray], dtype: str) -> Optional[np.ndarray]:
    """Exact widening of stored values (bf16 bits or f32) to float64."""
    if a is None:
        return None
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    return a.astype(np.float64)
