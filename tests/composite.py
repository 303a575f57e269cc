"""An independent float64 restatement of the projection with PyTorch CPU library ops.

Used only to pin the oracle. Each step is a library routine or textbook
identity rather than the oracle's own loops (and ``composite_backward``
differentiates it with ``torch.autograd``, pinning the oracle's backward):

* gather: ``torch.permute`` + ``reshape`` (the rearrange of "Make fused_ff_qkv
  contiguous", Walrus PR #12);
* fused linear: ``torch.addmm``;
* activations: ``torch.nn.functional.gelu`` (erf / tanh) and ``silu``;
* rotary embedding: multiplication of the complex number u[i] + i*u[i+half]
  by exp(i*theta) in complex128 (the rotate-half form of "Improve performance
  on RoPE", nvFuser issue #1597, written as a complex rotation);
* split: ``transpose(1, 2)`` then flattening batch and heads, the conversion to
  the [batch*heads, tokens, head_dim] layout of "Improve performance via
  batched-matmul and fused multiplies" (memory-efficient-attention issue #7);
  grouped-query heads follow the view/permute/split of the split_qkv listing.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np
import torch
import torch.nn.functional as Fn


def composite(x64: np.ndarray, W64: np.ndarray, b64: Optional[np.ndarray], **kw
              ) -> Dict[str, np.ndarray]:
    x = torch.from_numpy(np.asarray(x64, dtype=np.float64))
    Wt = torch.from_numpy(np.asarray(W64, dtype=np.float64))
    bt = None if b64 is None else torch.from_numpy(np.asarray(b64, dtype=np.float64))
    return {k: v.detach().contiguous().numpy() for k, v in _composite_t(x, Wt, bt, **kw).items()}


def composite_backward(x64: np.ndarray, W64: np.ndarray, b64: Optional[np.ndarray],
                       grads64: Dict[str, Optional[np.ndarray]], **kw) -> Dict[str, np.ndarray]:
    """Gradients of sum(g * output) by ``torch.autograd`` through the composite:
    dx [M, C] in token order, dW [C, N], db [N] (zeros when there is no bias)."""
    x = torch.from_numpy(np.asarray(x64, dtype=np.float64)).requires_grad_(True)
    Wt = torch.from_numpy(np.asarray(W64, dtype=np.float64)).requires_grad_(True)
    bt = torch.zeros(Wt.shape[1], dtype=torch.float64, requires_grad=True) if b64 is None else \
        torch.from_numpy(np.asarray(b64, dtype=np.float64)).requires_grad_(True)
    out = _composite_t(x, Wt, bt, **kw)
    loss = sum((out[k] * torch.from_numpy(np.asarray(g, dtype=np.float64))).sum()
               for k, g in grads64.items() if g is not None)
    dx, dW, db = torch.autograd.grad(loss, (x, Wt, bt))
    channel_dim = kw["channel_dim"]
    nd = x.dim()
    perm = [a for a in range(nd) if a != channel_dim] + [channel_dim]
    return {"dx": dx.permute(*perm).reshape(-1, x.shape[channel_dim]).numpy(),
            "dW": dW.numpy(), "db": db.numpy()}


def _composite_t(x: torch.Tensor, Wt: torch.Tensor, bt: Optional[torch.Tensor], *,
                 channel_dim: int, n_batch_dims: int, C: int, F: int, heads: int, head_dim: int,
                 act: int, rope_base: float, pos: Optional[np.ndarray] = None, groups: int = 0,
                 rope_n_elem: int = 0, k_transposed: bool = False,
                 rope_cos: Optional[np.ndarray] = None,
                 rope_sin: Optional[np.ndarray] = None) -> Dict[str, torch.Tensor]:
    nd = x.dim()
    perm = [a for a in range(nd) if a != channel_dim] + [channel_dim]
    tok = [x.shape[a] for a in range(nd) if a != channel_dim]
    Bb = int(np.prod(tok[:n_batch_dims], dtype=np.int64))
    T = int(np.prod(tok[n_batch_dims:], dtype=np.int64))
    M = Bb * T
    X = x.permute(*perm).reshape(M, C)
    if bt is None:
        bt = torch.zeros(Wt.shape[1], dtype=torch.float64)
    Y = torch.addmm(bt, X, Wt)
    ff = Y[:, :F]
    if act == 1:
        ff = Fn.gelu(ff, approximate="none")
    elif act == 2:
        ff = Fn.gelu(ff, approximate="tanh")
    elif act == 3:
        ff = Fn.silu(ff)
    elif act == 4:
        ff = torch.square(Fn.relu(ff))
    hd = head_dim
    rest = Y[:, F:]
    if groups:
        qpk = heads // groups
        qkv = rest.reshape(Bb, T, groups, qpk + 2, hd).permute(0, 2, 3, 1, 4)
        q, k, v = qkv.split((qpk, 1, 1), dim=2)
        q = q.reshape(Bb, heads, T, hd)
        k = k.reshape(Bb, groups, T, hd)
        v = v.reshape(Bb, groups, T, hd)
    else:
        q = rest[:, :C].reshape(Bb, T, heads, hd).transpose(1, 2)
        k = rest[:, C:2 * C].reshape(Bb, T, heads, hd).transpose(1, 2)
        v = rest[:, 2 * C:3 * C].reshape(Bb, T, heads, hd).transpose(1, 2)
    if rope_base > 0 and heads > 0:
        n = rope_n_elem or hd
        half = n // 2
        p = torch.arange(T, dtype=torch.float64) if pos is None else torch.from_numpy(
            np.asarray(pos, dtype=np.float64))
        inv = torch.tensor([rope_base ** (-2.0 * i / n) for i in range(half)], dtype=torch.float64)
        rot = torch.polar(torch.ones(T, half, dtype=torch.float64), p[:, None] * inv[None, :])

        def rope(u):
            z = torch.complex(u[..., :half], u[..., half:n]) * rot
            return torch.cat([z.real, z.imag, u[..., n:]], dim=-1)

        if rope_cos is not None:
            # caller tables, one cos/sin per rotated lane: the elementwise form
            # x*cos + cat(-x2, x1)*sin
            tc = torch.from_numpy(np.asarray(rope_cos, dtype=np.float64))
            ts = torch.from_numpy(np.asarray(rope_sin, dtype=np.float64))

            def rope(u):  # noqa: F811
                xr = u[..., :n]
                rotated = torch.cat([-xr[..., half:], xr[..., :half]], dim=-1)
                return torch.cat([xr * tc + rotated * ts, u[..., n:]], dim=-1)

        q, k = rope(q), rope(k)
    return {
        "ff": ff,
        "q": q.flatten(end_dim=1),
        "k": (k.transpose(-1, -2) if k_transposed else k).flatten(end_dim=1),
        "v": v.flatten(end_dim=1),
    }
