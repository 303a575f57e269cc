"""Fused input projection on one GB300 — Python binding of ``libfp.so``.

Argument marshalling only: every step of the projection runs in the library's
CUDA kernels. The functions below carry the names of the C ABI declared in
``include/fp.h``; ``FusedProjection`` wraps them for torch tensors (torch is
used for device memory and streams only).

If the library has not been built, ``load()`` raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence, Tuple

from . import _build

FP_OK = 0
FP_ERR_INVALID_ARG = 1
FP_ERR_UNSUPPORTED_LAYOUT = 2
FP_ERR_MISALIGNED = 3
FP_ERR_CUDA = 4
FP_ERR_OUT_OF_MEMORY = 5
FP_ERR_TIMEOUT = 6
FP_ERR_DEVICE_BOUNDS = 7

FP_ACT_NONE, FP_ACT_GELU_ERF, FP_ACT_GELU_TANH, FP_ACT_SILU, FP_ACT_RELU2 = 0, 1, 2, 3, 4
ACTS = {"none": 0, "gelu": 1, "gelu_erf": 1, "gelu_tanh": 2, "silu": 3, "relu2": 4}
FP_BF16, FP_F32 = 0, 1
FP_MAX_DIMS = 8

FP_OPT_WAIT_LIMIT_NS = 1
FP_OPT_INJECT_STALL = 2
FP_OPT_GROUP_M = 3
FP_OPT_MAX_CTAS = 4
FP_OPT_CLUSTER = 5
FP_OPT_BOUNDS_CHECK = 6
FP_OPT_TILE_N = 7

# the C ABI's entry points, as declared in include/fp.h
EXPORTS = ("fp_create", "fp_create_ex", "fp_forward", "fp_forward_host", "fp_forward_rope_table",
           "fp_forward_noalloc", "fp_backward_workspace_size", "fp_backward", "fp_backward_host",
           "fp_attention",
           "fp_reserve", "fp_get_device_status",
           "fp_last_launch_count", "fp_status_string", "fp_last_error", "fp_set_option",
           "fp_destroy")


class fp_layout(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("sizes", ctypes.c_int64 * FP_MAX_DIMS), ("strides", ctypes.c_int64 * FP_MAX_DIMS),
                ("channel_dim", ctypes.c_int32), ("n_batch_dims", ctypes.c_int32)]


class fp_config(ctypes.Structure):
    _fields_ = [("C", ctypes.c_int32), ("ff_hidden", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_query_groups", ctypes.c_int32),
                ("rope_n_elem", ctypes.c_int32), ("act", ctypes.c_int32),
                ("rope_base", ctypes.c_float), ("k_transposed", ctypes.c_int32)]


class fp_rope_table(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int32), ("stride_t", ctypes.c_int64),
                ("stride_i", ctypes.c_int64)]


class FpError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"fp status {status}: {msg}")
        self.status = status


_lib = None


def library_path() -> str:
    return _build.LIB


def load():
    """Load libfp.so; raises if it is missing (build it with ``_build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"libfp.so not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.fp_create.argtypes = [ctypes.POINTER(P), I, I, I, I, I, ctypes.c_float]
    lib.fp_create.restype = I
    lib.fp_create_ex.argtypes = [ctypes.POINTER(P), ctypes.POINTER(fp_config)]
    lib.fp_create_ex.restype = I
    lib.fp_forward.argtypes = [P, P, ctypes.POINTER(fp_layout), P, P, P, P, P, P, P, P]
    lib.fp_forward.restype = I
    lib.fp_forward_host.argtypes = [P, P, ctypes.POINTER(fp_layout), P, P, P, P, P, P, P, P]
    lib.fp_forward_host.restype = I
    lib.fp_forward_rope_table.argtypes = [P, P, ctypes.POINTER(fp_layout), P, P, P, P,
                                          ctypes.POINTER(fp_rope_table), P, P, P, P, P]
    lib.fp_forward_rope_table.restype = I
    lib.fp_forward_noalloc.argtypes = [ctypes.POINTER(fp_config), P, ctypes.POINTER(fp_layout), P,
                                       P, P, P, P, P, P, P]
    lib.fp_forward_noalloc.restype = I
    lib.fp_backward_workspace_size.argtypes = [P, ctypes.POINTER(fp_layout),
                                               ctypes.POINTER(ctypes.c_size_t)]
    lib.fp_backward_workspace_size.restype = I
    lib.fp_backward.argtypes = [P, P, ctypes.POINTER(fp_layout), P, P, P, P, P, P, P, P, P, P, P,
                                ctypes.c_size_t, P]
    lib.fp_backward.restype = I
    lib.fp_backward_host.argtypes = [P, P, ctypes.POINTER(fp_layout), P, P, P, P, P, P, P, P, P,
                                     P, P]
    lib.fp_backward_host.restype = I
    lib.fp_attention.argtypes = [P, P, P, P, P, I64, I64, I64, ctypes.c_float, P]
    lib.fp_attention.restype = I
    lib.fp_reserve.argtypes = [P, I64]
    lib.fp_reserve.restype = I
    lib.fp_get_device_status.argtypes = [P, P]
    lib.fp_get_device_status.restype = I
    lib.fp_last_launch_count.argtypes = [P]
    lib.fp_last_launch_count.restype = I
    lib.fp_status_string.argtypes = [I]
    lib.fp_status_string.restype = ctypes.c_char_p
    lib.fp_last_error.argtypes = []
    lib.fp_last_error.restype = ctypes.c_char_p
    lib.fp_set_option.argtypes = [P, I, I64]
    lib.fp_set_option.restype = I
    lib.fp_destroy.argtypes = [P]
    lib.fp_destroy.restype = None
    _lib = lib
    return lib


# ----------------------------------------------------------------- C-ABI mirrors

def fp_status_string(status: int) -> str:
    return load().fp_status_string(status).decode()


def fp_last_error() -> str:
    return load().fp_last_error().decode()


def fp_create(C: int, ff_hidden: int, heads: int, head_dim: int, act: int,
              rope_base: float) -> Tuple[int, Optional[int]]:
    """Returns (status, plan handle or None)."""
    h = ctypes.c_void_p()
    st = load().fp_create(ctypes.byref(h), C, ff_hidden, heads, head_dim, act, rope_base)
    return st, (h.value if st == FP_OK else None)


def fp_create_ex(config: fp_config) -> Tuple[int, Optional[int]]:
    """Returns (status, plan handle or None)."""
    h = ctypes.c_void_p()
    st = load().fp_create_ex(ctypes.byref(h), ctypes.byref(config))
    return st, (h.value if st == FP_OK else None)


def fp_forward(plan: int, x: int, layout: fp_layout, W: int, b: Optional[int], pos: Optional[int],
               out_ff: Optional[int], out_q: Optional[int], out_k: Optional[int],
               out_v: Optional[int], stream: Optional[int]) -> int:
    return load().fp_forward(plan, x, ctypes.byref(layout), W, b, pos, out_ff, out_q, out_k, out_v,
                             stream)


def fp_forward_host(plan: int, x_host: int, layout: fp_layout, W: int, b: Optional[int],
                    pos: Optional[int], out_ff: Optional[int], out_q: Optional[int],
                    out_k: Optional[int], out_v: Optional[int], stream: Optional[int]) -> int:
    """fp_forward on page-locked host x and outputs (copies pipelined in the library)."""
    return load().fp_forward_host(plan, x_host, ctypes.byref(layout), W, b, pos, out_ff, out_q,
                                  out_k, out_v, stream)


def fp_forward_rope_table(plan: int, x: int, layout: fp_layout, W: int, b: Optional[int],
                          rope_cos: int, rope_sin: int, table: fp_rope_table,
                          out_ff: Optional[int], out_q: Optional[int], out_k: Optional[int],
                          out_v: Optional[int], stream: Optional[int]) -> int:
    return load().fp_forward_rope_table(plan, x, ctypes.byref(layout), W, b, rope_cos, rope_sin,
                                        ctypes.byref(table), out_ff, out_q, out_k, out_v, stream)


def fp_forward_noalloc(config: fp_config, x: int, layout: fp_layout, W: int, b: Optional[int],
                       pos: Optional[int], out_ff: Optional[int], out_q: Optional[int],
                       out_k: Optional[int], out_v: Optional[int], stream: Optional[int]) -> int:
    """fp_forward without a plan and without any device allocation (static scratch)."""
    return load().fp_forward_noalloc(ctypes.byref(config), x, ctypes.byref(layout), W, b, pos,
                                     out_ff, out_q, out_k, out_v, stream)


def fp_backward_workspace_size(plan: int, layout: fp_layout) -> Tuple[int, int]:
    n = ctypes.c_size_t(0)
    st = load().fp_backward_workspace_size(plan, ctypes.byref(layout), ctypes.byref(n))
    return st, n.value


def fp_backward(plan: int, x: int, layout: fp_layout, W: int, b: Optional[int],
                pos: Optional[int], g_ff: Optional[int], g_q: Optional[int], g_k: Optional[int],
                g_v: Optional[int], dx: int, dW: int, db: Optional[int], workspace: int,
                workspace_bytes: int, stream: Optional[int]) -> int:
    return load().fp_backward(plan, x, ctypes.byref(layout), W, b, pos, g_ff, g_q, g_k, g_v, dx,
                              dW, db, workspace, workspace_bytes, stream)


def fp_backward_host(plan: int, x: int, layout: fp_layout, W: int, b: Optional[int],
                     pos: Optional[int], g_ff: Optional[int], g_q: Optional[int],
                     g_k: Optional[int], g_v: Optional[int], dx: int, dW: int,
                     db: Optional[int], stream: Optional[int]) -> int:
    """fp_backward on page-locked host x, gradients and results (copies pipelined)."""
    return load().fp_backward_host(plan, x, ctypes.byref(layout), W, b, pos, g_ff, g_q, g_k, g_v,
                                   dx, dW, db, stream)


def fp_attention(plan: int, q: int, k: int, v: int, out: int, batch: int, T_q: int, T_k: int,
                 scale: float, stream: Optional[int]) -> int:
    return load().fp_attention(plan, q, k, v, out, batch, T_q, T_k, scale, stream)


def fp_reserve(plan: int, max_tokens_per_batch: int) -> int:
    return load().fp_reserve(plan, max_tokens_per_batch)


def fp_get_device_status(plan: Optional[int], stream: Optional[int]) -> int:
    """plan None: the status words of fp_forward_noalloc on the current device."""
    return load().fp_get_device_status(plan, stream)


def fp_last_launch_count(plan: int) -> int:
    return load().fp_last_launch_count(plan)


def fp_set_option(plan: int, opt: int, value: int) -> int:
    return load().fp_set_option(plan, opt, value)


def fp_destroy(plan: Optional[int]) -> None:
    if plan:
        load().fp_destroy(plan)


def make_layout(sizes: Sequence[int], strides: Sequence[int], channel_dim: int, n_batch_dims: int,
                dtype: int) -> fp_layout:
    L = fp_layout()
    L.dtype = dtype
    L.ndim = len(sizes)
    for i, (s, st) in enumerate(zip(sizes, strides)):
        L.sizes[i] = int(s)
        L.strides[i] = int(st)
    L.channel_dim = channel_dim
    L.n_batch_dims = n_batch_dims
    return L


def check(status: int) -> None:
    if status != FP_OK:
        raise FpError(status, f"{fp_status_string(status)}: {fp_last_error()}")


# ----------------------------------------------------------------- torch wrapper

class FusedProjection:
    """A plan plus torch-tensor marshalling.

    ``forward(x, W, b, pos)`` returns ``(ff, q, k, v)`` (None for empty
    blocks), allocated on x's device with x's dtype; the work is enqueued on
    torch's current stream of that device.
    """

    def __init__(self, C: int, ff_hidden: int, heads: int, head_dim: int, act="none",
                 rope_base: float = 0.0, n_query_groups: int = 0, rope_n_elem: int = 0,
                 k_transposed: bool = False):
        a = ACTS[act] if isinstance(act, str) else int(act)
        cfg = fp_config(C, ff_hidden, heads, head_dim, n_query_groups, rope_n_elem, a,
                        float(rope_base), int(bool(k_transposed)))
        self.k_transposed = bool(k_transposed) and heads > 0
        st, h = fp_create_ex(cfg)
        check(st)
        self.plan = h
        self.C, self.F, self.heads, self.head_dim = C, ff_hidden, heads, head_dim
        self.kv_heads = n_query_groups if n_query_groups else heads
        self.N = ff_hidden + (heads + 2 * self.kv_heads) * head_dim

    def close(self):
        if getattr(self, "plan", None):
            fp_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_option(self, opt: int, value: int) -> None:
        check(fp_set_option(self.plan, opt, value))

    def reserve(self, max_tokens_per_batch: int) -> None:
        check(fp_reserve(self.plan, max_tokens_per_batch))

    def device_status(self, stream=None) -> int:
        import torch
        s = torch.cuda.current_stream().cuda_stream if stream is None else stream
        return fp_get_device_status(self.plan, s)

    @property
    def last_launch_count(self) -> int:
        return fp_last_launch_count(self.plan)

    def _head_shape(self, Bb: int, nh: int, T: int, transposed: bool):
        return (Bb * nh, self.head_dim, T) if transposed else (Bb * nh, T, self.head_dim)

    def out_shapes(self, x_shape: Sequence[int], channel_dim: int, n_batch_dims: int):
        tok = [s for a, s in enumerate(x_shape) if a != channel_dim]
        Bb = 1
        for s in tok[:n_batch_dims]:
            Bb *= s
        T = 1
        for s in tok[n_batch_dims:]:
            T *= s
        return Bb, T

    def forward(self, x, W, b=None, pos=None, *, channel_dim: int, n_batch_dims: int = 1,
                out=None, stream=None, rope_cos=None, rope_sin=None):
        """rope_cos/rope_sin: optional [T, n_rot] tables (any strides) used per lane
        instead of positions."""
        import torch
        if x.dtype not in (torch.bfloat16, torch.float32):
            raise TypeError(f"x must be bfloat16 or float32, got {x.dtype}")
        dt = FP_BF16 if x.dtype == torch.bfloat16 else FP_F32
        Bb, T = self.out_shapes(x.shape, channel_dim, n_batch_dims)
        M = Bb * T
        # the C ABI sees raw pointers: check the buffer sizes here
        if tuple(W.shape) != (self.C, self.N) or not W.is_contiguous() or W.dtype != x.dtype:
            raise ValueError(f"W must be a contiguous [{self.C}, {self.N}] {x.dtype} tensor, "
                             f"got {tuple(W.shape)} {W.dtype}")
        if b is not None and (tuple(b.shape) != (self.N,) or not b.is_contiguous()
                              or b.dtype != x.dtype):
            raise ValueError(f"b must be a contiguous [{self.N}] {x.dtype} tensor")
        if pos is not None and (tuple(pos.shape) != (T,) or pos.dtype != torch.int32
                                or not pos.is_contiguous()):
            raise ValueError(f"pos must be a contiguous int32 [{T}] tensor")
        for t in (W, b, pos):
            if t is not None and t.device != x.device:
                raise ValueError("all tensors must be on x's device")
        if out is None:
            ff = torch.empty((M, self.F), device=x.device, dtype=x.dtype) if self.F else None
            qkv = [torch.empty(self._head_shape(Bb, nh, T, kt), device=x.device, dtype=x.dtype)
                   for nh, kt in ((self.heads, False), (self.kv_heads, self.k_transposed),
                                  (self.kv_heads, False))] \
                if self.heads else [None, None, None]
            out = (ff, *qkv)
        else:
            want = [(M, self.F) if self.F else None] + \
                   [self._head_shape(Bb, nh, T, kt) if self.heads else None
                    for nh, kt in ((self.heads, False), (self.kv_heads, self.k_transposed),
                                   (self.kv_heads, False))]
            for o, shp in zip(out, want):
                if (o is None) != (shp is None) or (o is not None and (
                        tuple(o.shape) != shp or not o.is_contiguous() or o.dtype != x.dtype)):
                    raise ValueError(f"output buffers must be contiguous {want}")
        L = make_layout(x.shape, x.stride(), channel_dim, n_batch_dims, dt)
        ptr = lambda t: None if t is None else t.data_ptr()
        if stream is None:
            stream = torch.cuda.current_stream(x.device).cuda_stream
        if rope_cos is not None or rope_sin is not None:
            if rope_cos is None or rope_sin is None or pos is not None:
                raise ValueError("give rope_cos and rope_sin together, without pos")
            if rope_cos.shape != rope_sin.shape or rope_cos.stride() != rope_sin.stride() or \
                    rope_cos.dim() != 2 or rope_cos.shape[0] != T or rope_cos.dtype != rope_sin.dtype \
                    or rope_cos.dtype not in (torch.bfloat16, torch.float32):
                raise ValueError("rope_cos/rope_sin must be matching [T, n_rot] bf16/f32 tensors")
            tl = fp_rope_table(FP_BF16 if rope_cos.dtype == torch.bfloat16 else FP_F32,
                               rope_cos.stride(0), rope_cos.stride(1))
            st = fp_forward_rope_table(self.plan, x.data_ptr(), L, W.data_ptr(), ptr(b),
                                       rope_cos.data_ptr(), rope_sin.data_ptr(), tl, ptr(out[0]),
                                       ptr(out[1]), ptr(out[2]), ptr(out[3]), stream)
        else:
            st = fp_forward(self.plan, x.data_ptr(), L, W.data_ptr(), ptr(b), ptr(pos),
                            ptr(out[0]), ptr(out[1]), ptr(out[2]), ptr(out[3]), stream)
        check(st)
        return out

    def forward_host(self, x, W, b=None, pos=None, *, channel_dim: int, n_batch_dims: int = 1,
                     out=None, stream=None, device=None):
        """The projection of a page-locked host x into page-locked host outputs
        (allocated here when out is None); W, b and pos live on the GPU. The
        library moves x and the outputs through device staging in chunks,
        overlapping the copies with the compute. Returns (ff, q, k, v) host
        tensors, complete once `stream` reaches the end of the call's work."""
        import torch
        if x.device.type != "cpu" or not x.is_pinned():
            raise ValueError("x must be a page-locked (pinned) CPU tensor")
        if x.dtype not in (torch.bfloat16, torch.float32):
            raise TypeError(f"x must be bfloat16 or float32, got {x.dtype}")
        dev = W.device if device is None else torch.device(device)
        dt = FP_BF16 if x.dtype == torch.bfloat16 else FP_F32
        Bb, T = self.out_shapes(x.shape, channel_dim, n_batch_dims)
        M = Bb * T
        if tuple(W.shape) != (self.C, self.N) or not W.is_contiguous() or W.dtype != x.dtype \
                or W.device.type != "cuda":
            raise ValueError(f"W must be a contiguous [{self.C}, {self.N}] {x.dtype} CUDA tensor")
        if b is not None and (tuple(b.shape) != (self.N,) or not b.is_contiguous()
                              or b.dtype != x.dtype or b.device != W.device):
            raise ValueError(f"b must be a contiguous [{self.N}] {x.dtype} tensor on W's device")
        if pos is not None and (tuple(pos.shape) != (T,) or pos.dtype != torch.int32
                                or not pos.is_contiguous() or pos.device != W.device):
            raise ValueError(f"pos must be a contiguous int32 [{T}] tensor on W's device")
        want = [(M, self.F) if self.F else None] + \
               [self._head_shape(Bb, nh, T, kt) if self.heads else None
                for nh, kt in ((self.heads, False), (self.kv_heads, self.k_transposed),
                               (self.kv_heads, False))]
        if out is None:
            out = tuple(None if shp is None else torch.empty(shp, dtype=x.dtype, pin_memory=True)
                        for shp in want)
        for o, shp in zip(out, want):
            if (o is None) != (shp is None) or (o is not None and (
                    tuple(o.shape) != shp or not o.is_contiguous() or o.dtype != x.dtype
                    or o.device.type != "cpu" or not o.is_pinned())):
                raise ValueError(f"output buffers must be contiguous pinned CPU tensors {want}")
        L = make_layout(x.shape, x.stride(), channel_dim, n_batch_dims, dt)
        ptr = lambda t: None if t is None else t.data_ptr()
        if stream is None:
            stream = torch.cuda.current_stream(dev).cuda_stream
        with torch.cuda.device(dev):
            st = fp_forward_host(self.plan, x.data_ptr(), L, W.data_ptr(), ptr(b), ptr(pos),
                                 ptr(out[0]), ptr(out[1]), ptr(out[2]), ptr(out[3]), stream)
        check(st)
        return out

    def attention(self, q, k, v, *, batch: int, scale: float = 0.0, out=None, stream=None):
        """Softmax attention over this plan's q, k, v outputs (k pre-transposed when
        the plan emits it so). Returns out [batch*heads, T_q, head_dim], bf16, on
        torch's current stream."""
        import torch
        for t in (q, k, v):
            if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.device != q.device:
                raise ValueError("q, k, v must be contiguous bfloat16 tensors on one device")
        hd = self.head_dim
        if q.dim() != 3 or q.shape[0] != batch * self.heads or q.shape[2] != hd:
            raise ValueError(f"q must be [{batch * self.heads}, T_q, {hd}]")
        T_q = q.shape[1]
        kvn = batch * self.kv_heads
        T_k = v.shape[1]
        k_want = (kvn, hd, T_k) if self.k_transposed else (kvn, T_k, hd)
        if tuple(v.shape) != (kvn, T_k, hd) or tuple(k.shape) != k_want:
            raise ValueError(f"k must be {k_want} and v {(kvn, T_k, hd)}")
        if out is None:
            out = torch.empty_like(q)
        elif tuple(out.shape) != tuple(q.shape) or not out.is_contiguous() or out.dtype != q.dtype:
            raise ValueError("out must be a contiguous tensor shaped like q")
        if stream is None:
            stream = torch.cuda.current_stream(q.device).cuda_stream
        check(fp_attention(self.plan, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           batch, T_q, T_k, scale, stream))
        return out

    def backward(self, x, W, b, grads, pos=None, *, channel_dim: int, n_batch_dims: int = 1,
                  dx=None, workspace=None, stream=None):
        """Gradients of ``forward``'s outputs: ``grads`` = (g_ff, g_q, g_k, g_v) in the
        output layouts (None where the output is None). Returns ``(dx, dW, db)``: dx
        laid out like x (x's strides), dW float32 [C, N], db float32 [N] (None
        without bias). The work is enqueued on torch's current stream."""
        import torch
        if x.dtype != torch.bfloat16:
            raise TypeError("the backward takes bfloat16 activations")
        Bb, T = self.out_shapes(x.shape, channel_dim, n_batch_dims)
        M = Bb * T
        if tuple(W.shape) != (self.C, self.N) or not W.is_contiguous() or W.dtype != x.dtype:
            raise ValueError(f"W must be a contiguous [{self.C}, {self.N}] {x.dtype} tensor")
        if b is not None and (tuple(b.shape) != (self.N,) or not b.is_contiguous()
                              or b.dtype != x.dtype):
            raise ValueError(f"b must be a contiguous [{self.N}] {x.dtype} tensor")
        if pos is not None and (tuple(pos.shape) != (T,) or pos.dtype != torch.int32
                                or not pos.is_contiguous()):
            raise ValueError(f"pos must be a contiguous int32 [{T}] tensor")
        want = [(M, self.F) if self.F else None] + \
               [self._head_shape(Bb, nh, T, kt) if self.heads else None
                for nh, kt in ((self.heads, False), (self.kv_heads, self.k_transposed),
                               (self.kv_heads, False))]
        grads = tuple(grads)
        for g, shp in zip(grads, want):
            if (g is None) != (shp is None) or (g is not None and (
                    tuple(g.shape) != shp or not g.is_contiguous() or g.dtype != x.dtype
                    or g.device != x.device)):
                raise ValueError(f"gradients must be contiguous {want} on x's device")
        if dx is None:
            dx = torch.empty_strided(x.shape, x.stride(), dtype=x.dtype, device=x.device)
        elif tuple(dx.shape) != tuple(x.shape) or dx.stride() != x.stride() or dx.dtype != x.dtype:
            raise ValueError("dx must have x's shape, strides and dtype")
        dW = torch.empty((self.C, self.N), dtype=torch.float32, device=x.device)
        db = torch.empty((self.N,), dtype=torch.float32, device=x.device) if b is not None else None
        L = make_layout(x.shape, x.stride(), channel_dim, n_batch_dims, FP_BF16)
        st, need = fp_backward_workspace_size(self.plan, L)
        check(st)
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty((need,), dtype=torch.uint8, device=x.device)
        ptr = lambda t: None if t is None else t.data_ptr()
        if stream is None:
            stream = torch.cuda.current_stream(x.device).cuda_stream
        check(fp_backward(self.plan, x.data_ptr(), L, W.data_ptr(), ptr(b), ptr(pos), ptr(grads[0]),
                          ptr(grads[1]), ptr(grads[2]), ptr(grads[3]), dx.data_ptr(), dW.data_ptr(),
                          ptr(db), workspace.data_ptr(),
                          workspace.numel() * workspace.element_size(), stream))
        return dx, dW, db

    def backward_host(self, x, W, b, grads, pos=None, *, channel_dim: int, n_batch_dims: int = 1,
                      out=None, stream=None):
        """``backward`` on a page-locked host x and host gradients: returns host
        ``(dx, dW, db)`` (page-locked; allocated here when out is None). W, b and
        pos live on the GPU; x must be dense. The library moves the data in batch
        chunks, overlapping the copies with the compute."""
        import torch
        if x.device.type != "cpu" or not x.is_pinned() or not x.is_contiguous():
            raise ValueError("x must be a contiguous page-locked (pinned) CPU tensor")
        if x.dtype != torch.bfloat16:
            raise TypeError("the backward takes bfloat16 activations")
        Bb, T = self.out_shapes(x.shape, channel_dim, n_batch_dims)
        M = Bb * T
        if tuple(W.shape) != (self.C, self.N) or not W.is_contiguous() or W.dtype != x.dtype \
                or W.device.type != "cuda":
            raise ValueError(f"W must be a contiguous [{self.C}, {self.N}] {x.dtype} CUDA tensor")
        if b is not None and (tuple(b.shape) != (self.N,) or not b.is_contiguous()
                              or b.dtype != x.dtype or b.device != W.device):
            raise ValueError(f"b must be a contiguous [{self.N}] {x.dtype} tensor on W's device")
        if pos is not None and (tuple(pos.shape) != (T,) or pos.dtype != torch.int32
                                or not pos.is_contiguous() or pos.device != W.device):
            raise ValueError(f"pos must be a contiguous int32 [{T}] tensor on W's device")
        want = [(M, self.F) if self.F else None] + \
               [self._head_shape(Bb, nh, T, kt) if self.heads else None
                for nh, kt in ((self.heads, False), (self.kv_heads, self.k_transposed),
                               (self.kv_heads, False))]
        grads = tuple(grads)
        for g, shp in zip(grads, want):
            if (g is None) != (shp is None) or (g is not None and (
                    tuple(g.shape) != shp or not g.is_contiguous() or g.dtype != x.dtype
                    or g.device.type != "cpu" or not g.is_pinned())):
                raise ValueError(f"gradients must be contiguous pinned CPU tensors {want}")
        if out is None:
            out = (torch.empty_like(x).pin_memory(),
                   torch.empty((self.C, self.N), dtype=torch.float32).pin_memory(),
                   torch.empty((self.N,), dtype=torch.float32).pin_memory()
                   if b is not None else None)
        dx, dW, db = out
        for t, shp, dt in ((dx, tuple(x.shape), x.dtype), (dW, (self.C, self.N), torch.float32),
                           (db, (self.N,), torch.float32)):
            if t is not None and (tuple(t.shape) != shp or t.dtype != dt or not t.is_contiguous()
                                  or t.device.type != "cpu" or not t.is_pinned()):
                raise ValueError("dx, dW and db must be contiguous pinned CPU tensors")
        L = make_layout(x.shape, x.stride(), channel_dim, n_batch_dims, FP_BF16)
        ptr = lambda t: None if t is None else t.data_ptr()
        if stream is None:
            stream = torch.cuda.current_stream(W.device).cuda_stream
        with torch.cuda.device(W.device):
            check(fp_backward_host(self.plan, x.data_ptr(), L, W.data_ptr(), ptr(b), ptr(pos),
                                   ptr(grads[0]), ptr(grads[1]), ptr(grads[2]), ptr(grads[3]),
                                   dx.data_ptr(), dW.data_ptr(), ptr(db), stream))
        return dx, dW, db

