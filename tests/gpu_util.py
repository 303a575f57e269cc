"""Helpers shared by the GPU tests: moving generated inputs to the device,
running the library, and the tolerance rule."""
from __future__ import annotations

from typing import Dict, Optional, Sequence

import numpy as np
import torch

import ff_input_projection_gb300 as fpx
import fpsynth

# |gpu - ref| <= max(REL * |ref|, FLOOR * rms(ref over the whole output buffer))
TOL = {"bf16": (1e-2, 2e-2), "f32": (1e-4, 2e-4)}


def to_device(a: Optional[np.ndarray], dtype: str, device="cuda") -> Optional[torch.Tensor]:
    if a is None:
        return None
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(device)


def run(w: fpsynth.Workload, inp: Dict[str, np.ndarray], x_dev: Optional[torch.Tensor] = None,
        proj: Optional[fpx.FusedProjection] = None, pos: Optional[np.ndarray] = None):
    """Run the library on workload ``w``. ``x_dev`` may be a strided view to read in place."""
    if proj is None:
        proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base,
                                   w.n_query_groups, w.rope_n_elem, w.k_transposed)
    x = to_device(inp["x"], w.dtype) if x_dev is None else x_dev
    W = to_device(inp["W"], w.dtype)
    b = to_device(inp["b"], w.dtype)
    p = pos if pos is not None else inp.get("pos")
    pos_t = None if p is None else torch.from_numpy(np.ascontiguousarray(p, dtype=np.int32)).cuda()
    out = proj.forward(x, W, b, pos_t, channel_dim=w.channel_dim, n_batch_dims=w.n_batch_dims,
                       out=nan_outputs(proj, w, x.device))
    torch.cuda.synchronize()
    st = proj.device_status()
    assert st == fpx.FP_OK, fpx.fp_last_error()
    return dict(zip(("ff", "q", "k", "v"), out))


def out_shapes(proj: fpx.FusedProjection, w: fpsynth.Workload):
    """Shapes of (ff, q, k, v) for workload ``w`` (None for an empty block)."""
    Bb, T = proj.out_shapes(w.x_shape, w.channel_dim, w.n_batch_dims)
    ff = (Bb * T, proj.F) if proj.F else None
    if not proj.heads:
        return [ff, None, None, None]
    return [ff, proj._head_shape(Bb, proj.heads, T, False),
            proj._head_shape(Bb, proj.kv_heads, T, proj.k_transposed),
            proj._head_shape(Bb, proj.kv_heads, T, False)]


def nan_outputs(proj: fpx.FusedProjection, w: fpsynth.Workload, device="cuda"):
    """Output buffers filled with NaN: an element the kernels never write stays
    NaN and fails every comparison."""
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    return tuple(None if s is None else torch.full(s, float("nan"), dtype=dt, device=device)
                 for s in out_shapes(proj, w))


def host(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    return None if t is None else t.float().cpu().numpy().astype(np.float64)


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str,
                 rms: Optional[float] = None) -> None:
    rel, floor = TOL[dtype]
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if ref.size == 0:
        return
    if rms is None:
        rms = float(np.sqrt(np.mean(ref ** 2)))
    tol = np.maximum(rel * np.abs(ref), floor * rms)
    err = np.abs(got - ref)
    bad = ~(err <= tol)  # NaN (an element never written) counts as bad
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; worst err "
            f"{np.nanmax(err) if np.isfinite(err).any() else float('nan'):.3e} (rms {rms:.3e}); "
            f"first bad {idx.tolist()} "
            f"got {got[tuple(idx[0])]:.6f} ref {ref[tuple(idx[0])]:.6f}")
