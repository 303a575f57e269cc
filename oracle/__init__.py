"""CPU oracle of the fused input projection — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product library does not, and shares
no code with it. ``fp_oracle.c`` holds the definition (fp64, one token at a
time, following the pages' steps); this module builds it with gcc and calls it
through ctypes.

Parity pins: every function of the oracle is pinned by ``tests/test_oracle_pins.py``
(library cross-checks, closed forms, invariants, brute force, planted mistakes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "attn_oracle.c")]
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

ACT_NONE, ACT_GELU_ERF, ACT_GELU_TANH, ACT_SILU, ACT_RELU2 = 0, 1, 2, 3, 4

MUTATIONS = {
    "drop_bias": 1, "rope_sign": 2, "w_transposed": 3, "tanh_const": 4, "scatter_order": 5,
    "rope_interleaved": 6, "rope_freq": 7, "view_not_permute": 8, "act_on_q": 9,
    "pos_global": 10, "rope_on_v": 11, "qk_swapped": 12, "gelu_scale": 13,
    "relu2_unsquared": 14,
}
# planted mistakes of the attention oracle
ATTN_MUTATIONS = {"no_merge_rescale": 1, "no_scale": 2, "k_index_swap": 3,
                  "softmax_over_queries": 4, "sum_not_rescaled": 5}
# planted mistakes of the backward
BWD_MUTATIONS = {
    "bwd_rope_forward": 21, "bwd_act_value": 22, "bwd_no_recompute_bias": 23,
    "bwd_dw_swap": 24, "bwd_dx_no_w": 25,
}


def build(force: bool = False) -> str:
    """Compile fp_oracle.c into liboracle.so (plain C, no CUDA)."""
    if (not force and os.path.exists(_LIB)
            and all(os.path.getmtime(_LIB) >= os.path.getmtime(f) for f in _SRCS)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           *_SRCS, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        f = lib.oracle_forward
        f.restype = ctypes.c_int
        P = ctypes.c_void_p
        I = ctypes.c_int
        I64 = ctypes.c_int64
        f.argtypes = [P, I, I, P, P, I, I, P, P, P, P, P, I, I, I, I, I, I, I, I,
                      ctypes.c_double, P, I64, P, P, P, P, I, I]
        g = lib.oracle_backward
        g.restype = ctypes.c_int
        g.argtypes = [P, I, I, P, P, I, I, P, P, P, P, P, I, I, I, I, I, I, I, I,
                      ctypes.c_double, P, P, P, P, I, P, I64, P, I64, P, P, P, I, I]
        h = lib.oracle_attention
        h.restype = ctypes.c_int
        h.argtypes = [P, P, P, I, I64, I64, I64, I, I, ctypes.c_double, I64, I64, P, I, I]
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def forward(x: np.ndarray, W: np.ndarray, b: Optional[np.ndarray], *, channel_dim: int,
            n_batch_dims: int, C: int, F: int, heads: int, head_dim: int, act: int,
            rope_base: float, dtype: str, pos: Optional[np.ndarray] = None,
            rope_cos: Optional[np.ndarray] = None, rope_sin: Optional[np.ndarray] = None,
            groups: int = 0, rope_n_elem: int = 0, k_transposed: bool = False,
            rows: Optional[Sequence[int]] = None,
            threads: Optional[int] = None, mutate: int = 0,
            x_strides: Optional[Sequence[int]] = None, x_base: Optional[np.ndarray] = None
            ) -> Dict[str, np.ndarray]:
    """Evaluate the projection in fp64.

    ``x`` holds stored values (uint16 bf16 bits or float32) with logical shape
    ``x.shape``; by default it is addressed through its own (element) strides.
    To describe a strided view, pass the backing buffer as ``x_base`` and the
    element strides as ``x_strides``.

    Returns ``ff`` [M, F], ``q`` [B*heads, T, hd], ``k``/``v`` [B*kv, T, hd]
    (``k`` [B*kv, hd, T] with ``k_transposed``) when ``rows`` is None, else per-row arrays ``ff`` [R, F], ``q`` [R, heads*hd],
    ``k``/``v`` [R, kv*hd] for the requested token indices.
    """
    lib = _load()
    is_bf16 = dtype == "bf16"
    want = np.uint16 if is_bf16 else np.float32
    sizes = np.array(x.shape, dtype=np.int64)
    if x_base is None:
        xb = np.ascontiguousarray(x)
        if xb.dtype != want:
            raise TypeError(f"x must be {want}")
        strides = np.array([s // xb.itemsize for s in xb.strides], dtype=np.int64)
    else:
        xb = x_base
        if xb.dtype != want:
            raise TypeError(f"x_base must be {want}")
        strides = np.array(x_strides, dtype=np.int64)
    Wc = np.ascontiguousarray(W, dtype=want)
    bc = None if b is None else np.ascontiguousarray(b, dtype=want)
    posc = None if pos is None else np.ascontiguousarray(pos, dtype=np.int32)
    # caller tables: [T, n_rot] values, widened exactly to float64
    tcos = None if rope_cos is None else np.ascontiguousarray(rope_cos, dtype=np.float64)
    tsin = None if rope_sin is None else np.ascontiguousarray(rope_sin, dtype=np.float64)
    if (tcos is None) != (tsin is None):
        raise ValueError("rope_cos and rope_sin go together")
    nkv = groups if groups else heads
    tok = [s for a, s in enumerate(x.shape) if a != channel_dim]
    Bb = int(np.prod(tok[:n_batch_dims], dtype=np.int64))
    T = int(np.prod(tok[n_batch_dims:], dtype=np.int64))
    M = Bb * T
    if rows is None:
        kshape = (Bb * nkv, head_dim, T) if k_transposed else (Bb * nkv, T, head_dim)
        out = {"ff": np.zeros((M, F)), "q": np.zeros((Bb * heads, T, head_dim)),
               "k": np.zeros(kshape), "v": np.zeros((Bb * nkv, T, head_dim))}
        rr = None
        R = 0
    else:
        rr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        R = len(rr)
        out = {"ff": np.zeros((R, F)), "q": np.zeros((R, heads * head_dim)),
               "k": np.zeros((R, nkv * head_dim)), "v": np.zeros((R, nkv * head_dim))}
    if threads is None:
        threads = os.cpu_count() or 1
    rc = lib.oracle_forward(_ptr(xb), int(is_bf16), x.ndim, _ptr(sizes), _ptr(strides), channel_dim,
                            n_batch_dims, _ptr(Wc), _ptr(bc), _ptr(posc), _ptr(tcos), _ptr(tsin),
                            C, F, heads, head_dim,
                            groups, rope_n_elem, act, int(bool(k_transposed)), float(rope_base),
                            _ptr(rr), R,
                            _ptr(out["ff"]), _ptr(out["q"]), _ptr(out["k"]), _ptr(out["v"]),
                            int(threads), int(mutate))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out


def forward_workload(w, inputs: Dict[str, np.ndarray], **kw) -> Dict[str, np.ndarray]:
    """``forward`` with the shape parameters of an ``fpsynth.Workload``."""
    return forward(inputs["x"], inputs["W"], inputs["b"], channel_dim=w.channel_dim,
                   n_batch_dims=w.n_batch_dims, C=w.C, F=w.F, heads=w.heads,
                   head_dim=w.head_dim, act=w.act, rope_base=w.rope_base, dtype=w.dtype,
                   pos=inputs.get("pos"), rope_cos=inputs.get("rope_cos"),
                   rope_sin=inputs.get("rope_sin"), groups=w.n_query_groups,
                   rope_n_elem=w.rope_n_elem, k_transposed=w.k_transposed, **kw)


def backward(x: np.ndarray, W: np.ndarray, b: Optional[np.ndarray], grads: Dict[str, np.ndarray],
             *, channel_dim: int, n_batch_dims: int, C: int, F: int, heads: int, head_dim: int,
             act: int, rope_base: float, dtype: str, pos: Optional[np.ndarray] = None,
             rope_cos: Optional[np.ndarray] = None, rope_sin: Optional[np.ndarray] = None,
             groups: int = 0, rope_n_elem: int = 0, k_transposed: bool = False,
             rows: Optional[Sequence[int]] = None, cols: Optional[Sequence[int]] = None,
             threads: Optional[int] = None, mutate: int = 0) -> Dict[str, np.ndarray]:
    """Gradients of the projection in fp64, given upstream gradients ``grads``
    (keys ff, q, k, v; stored values in the forward's output layouts, dtype of x).

    Default: ``dx`` [M, C] (token order m = b*T + t), ``dW`` [C, N], ``db`` [N].
    With ``rows``: ``dx`` [R, C] of those tokens. With ``cols``: ``dW`` [C, K] and
    ``db`` [K] of those fused columns (summed over every token).
    """
    lib = _load()
    is_bf16 = dtype == "bf16"
    want = np.uint16 if is_bf16 else np.float32
    sizes = np.array(x.shape, dtype=np.int64)
    xb = np.ascontiguousarray(x)
    if xb.dtype != want:
        raise TypeError(f"x must be {want}")
    strides = np.array([s // xb.itemsize for s in xb.strides], dtype=np.int64)
    Wc = np.ascontiguousarray(W, dtype=want)
    bc = None if b is None else np.ascontiguousarray(b, dtype=want)
    posc = None if pos is None else np.ascontiguousarray(pos, dtype=np.int32)
    tcos = None if rope_cos is None else np.ascontiguousarray(rope_cos, dtype=np.float64)
    tsin = None if rope_sin is None else np.ascontiguousarray(rope_sin, dtype=np.float64)
    g = {k: (None if grads.get(k) is None else np.ascontiguousarray(grads[k], dtype=want))
         for k in ("ff", "q", "k", "v")}
    nkv = groups if groups else heads
    N = F + ((heads + 2 * groups) * head_dim if groups else 3 * heads * head_dim)
    tok = [s for a, s in enumerate(x.shape) if a != channel_dim]
    M = int(np.prod(tok, dtype=np.int64))
    if threads is None:
        threads = os.cpu_count() or 1
    rr = cc = None
    R = K = 0
    if rows is not None:
        mode = 1
        rr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        R = len(rr)
        out = {"dx": np.zeros((R, C))}
    elif cols is not None:
        mode = 2
        cc = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
        K = len(cc)
        out = {"dW": np.zeros((C, K)), "db": np.zeros(K)}
    else:
        mode = 0
        out = {"dx": np.zeros((M, C)), "dW": np.zeros((C, N)), "db": np.zeros(N)}
    del nkv
    rc = lib.oracle_backward(_ptr(xb), int(is_bf16), x.ndim, _ptr(sizes), _ptr(strides),
                             channel_dim, n_batch_dims, _ptr(Wc), _ptr(bc), _ptr(posc),
                             _ptr(tcos), _ptr(tsin), C, F, heads, head_dim, groups, rope_n_elem,
                             act, int(bool(k_transposed)), float(rope_base),
                             _ptr(g["ff"]), _ptr(g["q"]), _ptr(g["k"]), _ptr(g["v"]), mode,
                             _ptr(rr), R, _ptr(cc), K,
                             _ptr(out.get("dx")), _ptr(out.get("dW")), _ptr(out.get("db")),
                             int(threads), int(mutate))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out


def backward_workload(w, inputs: Dict[str, np.ndarray], grads: Dict[str, np.ndarray], **kw
                      ) -> Dict[str, np.ndarray]:
    """``backward`` with the shape parameters of an ``fpsynth.Workload``."""
    return backward(inputs["x"], inputs["W"], inputs["b"], grads, channel_dim=w.channel_dim,
                    n_batch_dims=w.n_batch_dims, C=w.C, F=w.F, heads=w.heads,
                    head_dim=w.head_dim, act=w.act, rope_base=w.rope_base, dtype=w.dtype,
                    pos=inputs.get("pos"), rope_cos=inputs.get("rope_cos"),
                    rope_sin=inputs.get("rope_sin"), groups=w.n_query_groups,
                    rope_n_elem=w.rope_n_elem, k_transposed=w.k_transposed, **kw)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, *, dtype: str,
              k_transposed: bool = False, scale: Optional[float] = None,
              q_chunk: Optional[int] = None, kv_chunk: Optional[int] = None,
              threads: Optional[int] = None, mutate: int = 0) -> np.ndarray:
    """Attention over the projection's outputs, in fp64 (attn_oracle.c).

    ``q`` [BH, Tq, hd], ``k`` [BH, Tk, hd] (or [BH, hd, Tk] with
    ``k_transposed``), ``v`` [BH, Tk, hd], stored values (uint16 bf16 bits or
    float32). ``scale`` defaults to hd**-0.5; ``q_chunk`` / ``kv_chunk`` default
    to one chunk (the page's fast paths). Returns [BH, Tq, hd] float64.
    """
    lib = _load()
    is_bf16 = dtype == "bf16"
    want = np.uint16 if is_bf16 else np.float32
    qc, kc, vc = (np.ascontiguousarray(a) for a in (q, k, v))
    for a in (qc, kc, vc):
        if a.dtype != want:
            raise TypeError(f"inputs must be {want}")
    BH, Tq, hd = qc.shape
    Tk = kc.shape[2] if k_transposed else kc.shape[1]
    if scale is None:
        scale = hd ** -0.5
    out = np.zeros((BH, Tq, hd))
    rc = lib.oracle_attention(_ptr(qc), _ptr(kc), _ptr(vc), int(is_bf16), BH, Tq, Tk, hd,
                              int(bool(k_transposed)), float(scale),
                              int(q_chunk or max(Tq, 1)), int(kv_chunk or Tk), _ptr(out),
                              int(threads or os.cpu_count() or 1), int(mutate))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out
