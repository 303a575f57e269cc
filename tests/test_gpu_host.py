"""fp_forward_host against the CPU oracle and against fp_forward, through the C
ABI (needs a GB300).

The host entry point splits the first batch axis of a dense x into up to 4
chunks and pipelines each chunk's upload, projection and download over two
staging slots. Cases: 2 chunks (tensor-core path, rotation, GELU ff), 3
uneven chunks over 5 batch elements, the fp32 FFMA path, a layout that is not
chunked (channel axis first) and a strided x (one chunk over the whole span),
two calls on different streams reusing the staging, and the rejection of
pageable host memory. Every output is compared with the oracle (the bf16 or
f32 tolerance rule) and bit for bit with fp_forward on the device, which runs
the same kernels on the same data.
"""
import numpy as np
import pytest
import torch

import ff_input_projection_gb300 as fpx
import fpsynth
import oracle
from tests.gpu_util import assert_close, host, run, to_device

pytestmark = pytest.mark.gpu

W_ = fpsynth.Workload
A = fpsynth

CASES = [
    # [2, 3, 64, 16, 16, 1] channels-first: 2 chunks of one batch element
    W_("host_walrus_small", (2, 3, 64, 16, 16, 1), 2, 1, 64, 128, 2, 32, A.ACT_GELU_ERF, 10000.0,
       True, "bf16", 91),
    # 5 batch elements: chunks of 2, 2 and 1
    W_("host_uneven", (5, 77, 192), 2, 1, 192, 0, 3, 64, A.ACT_NONE, 0.0, True, "bf16", 92),
    # fp32, NCHW: the FFMA kernel
    W_("host_fp32", (2, 32, 20, 20), 1, 1, 32, 64, 2, 16, A.ACT_SILU, 10000.0, True, "f32", 93),
    # channel axis first: not chunked, one copy of the whole x
    W_("host_channel_first_axis", (64, 2, 50), 0, 1, 64, 64, 2, 32, A.ACT_GELU_TANH, 10000.0,
       True, "bf16", 94),
    # grouped-query heads, partial rotary and k pre-transposed: 4 chunks whose
    # k/v ranges follow the group count
    W_("host_gqa_kt", (4, 130, 256), 2, 1, 256, 0, 8, 32, A.ACT_NONE, 10000.0, False, "bf16", 98,
       rope_n_elem=8, n_query_groups=2, k_transposed=True),
]


def pinned(a: np.ndarray, dtype: str) -> torch.Tensor:
    return to_device(a, dtype, device="cpu").pin_memory()


def host_run(w, inp, x_host=None, stream=None, proj=None):
    proj = proj or fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base,
                                       w.n_query_groups, w.rope_n_elem, w.k_transposed)
    x = pinned(inp["x"], w.dtype) if x_host is None else x_host
    W = to_device(inp["W"], w.dtype)
    b = to_device(inp["b"], w.dtype)
    out = proj.forward_host(x, W, b, None, channel_dim=w.channel_dim,
                            n_batch_dims=w.n_batch_dims, stream=stream)
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_OK
    return proj, dict(zip(("ff", "q", "k", "v"), out))


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_host_entry_matches_oracle_and_device_path(w, cuda_ok):
    inp = fpsynth.make_inputs(w)
    ref = oracle.forward_workload(w, inp)
    proj, out = host_run(w, inp)
    dev = run(w, inp)
    for k in ("ff", "q", "k", "v"):
        if out[k] is None:
            assert ref[k].size == 0
            continue
        assert out[k].device.type == "cpu"
        assert_close(host(out[k]), ref[k], w.dtype, f"{w.name}:{k}")
        assert torch.equal(out[k], dev[k].cpu()), f"{w.name}:{k} differs from fp_forward"


def test_host_entry_caller_positions(cuda_ok):
    """Caller positions: each chunk rebuilds the rotary table from them."""
    w = CASES[0]
    inp = fpsynth.make_inputs(w)
    pos = ((np.arange(w.T) * 37) % 1000 + 3).astype(np.int32)
    ref = oracle.forward_workload(w, {**inp, "pos": pos})
    proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base)
    out = proj.forward_host(pinned(inp["x"], w.dtype), to_device(inp["W"], w.dtype),
                            to_device(inp["b"], w.dtype), torch.from_numpy(pos).cuda(),
                            channel_dim=w.channel_dim, n_batch_dims=w.n_batch_dims)
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_OK
    for k, o in zip(("ff", "q", "k", "v"), out):
        assert_close(host(o), ref[k], w.dtype, f"pos:{k}")


def test_host_entry_launch_count(cuda_ok):
    """One projection per chunk: with the rotary table already built, 2 chunks
    launch twice what one device call on a chunk does."""
    w = CASES[0]
    inp = fpsynth.make_inputs(w)
    proj, _ = host_run(w, inp)  # builds the plan's table
    proj, _ = host_run(w, inp, proj=proj)
    host_launches = proj.last_launch_count
    x1 = to_device(inp["x"][:1], w.dtype)
    proj.forward(x1, to_device(inp["W"], w.dtype), to_device(inp["b"], w.dtype), None,
                 channel_dim=w.channel_dim, n_batch_dims=w.n_batch_dims)
    torch.cuda.synchronize()
    assert host_launches == 2 * proj.last_launch_count > 0


def test_host_entry_strided_x(cuda_ok):
    """A padded (non-dense) x goes up as one span and is read through its strides."""
    w = CASES[0]
    inp = fpsynth.make_inputs(w)
    ref = oracle.forward_workload(w, inp)
    x = to_device(inp["x"], w.dtype, device="cpu")
    big = torch.zeros((2, 4, 64, 16, 16, 1), dtype=x.dtype).pin_memory()
    big[:, :3] = x
    _, out = host_run(w, inp, x_host=big[:, :3])
    for k in ("ff", "q", "k", "v"):
        assert_close(host(out[k]), ref[k], w.dtype, f"strided:{k}")


def test_host_entry_two_streams_share_staging(cuda_ok):
    """Back-to-back calls on different streams: the second call's uploads wait
    for the first call's downloads, so both results are intact."""
    w = CASES[1]
    proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base)
    inps = [fpsynth.make_inputs(w)]
    w2 = W_(w.name, w.x_shape, w.channel_dim, w.n_batch_dims, w.C, w.F, w.heads, w.head_dim,
            w.act, w.rope_base, w.bias, w.dtype, 95)
    inps.append(fpsynth.make_inputs(w2))
    inps[1]["W"] = inps[0]["W"]
    inps[1]["b"] = inps[0]["b"]
    W = to_device(inps[0]["W"], w.dtype)
    b = to_device(inps[0]["b"], w.dtype)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for inp, s in zip(inps, streams):
        x = pinned(inp["x"], w.dtype)
        outs.append(proj.forward_host(x, W, b, None, channel_dim=w.channel_dim,
                                      n_batch_dims=w.n_batch_dims, stream=s.cuda_stream))
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_OK
    for inp, out in zip(inps, outs):
        ref = oracle.forward_workload(w, inp)
        for k, o in zip(("ff", "q", "k", "v"), out):
            if o is not None:
                assert_close(host(o), ref[k], w.dtype, f"two streams:{k}")


def test_host_entry_rejects_pageable_memory(cuda_ok):
    w = CASES[0]
    inp = fpsynth.make_inputs(w)
    proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base)
    x = to_device(inp["x"], w.dtype, device="cpu")  # pageable
    W = to_device(inp["W"], w.dtype)
    b = to_device(inp["b"], w.dtype)
    Bb, T = proj.out_shapes(w.x_shape, w.channel_dim, w.n_batch_dims)
    outs = [torch.empty((Bb * T, w.F), dtype=x.dtype).pin_memory()] + \
           [torch.empty((Bb * w.heads, T, w.head_dim), dtype=x.dtype).pin_memory()
            for _ in range(3)]
    L = fpx.make_layout(x.shape, x.stride(), w.channel_dim, w.n_batch_dims, fpx.FP_BF16)
    st = fpx.fp_forward_host(proj.plan, x.data_ptr(), L, W.data_ptr(), b.data_ptr(), None,
                             *[o.data_ptr() for o in outs], None)
    assert st == fpx.FP_ERR_INVALID_ARG
    assert "page-locked" in fpx.fp_last_error()
    xp = x.pin_memory()
    pageable_out = torch.empty_like(outs[0])
    st = fpx.fp_forward_host(proj.plan, xp.data_ptr(), L, W.data_ptr(), b.data_ptr(), None,
                             pageable_out.data_ptr(), *[o.data_ptr() for o in outs[1:]], None)
    assert st == fpx.FP_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        proj.forward_host(x, W, b, None, channel_dim=w.channel_dim, n_batch_dims=w.n_batch_dims)


BWD_CASES = [
    # channels-first, 2 chunks (dxᵀ kernel), GELU ff + rotated heads
    W_("bwd_host_walrus_small", (2, 3, 64, 16, 16, 1), 2, 1, 64, 128, 2, 32, A.ACT_GELU_ERF,
       10000.0, True, "bf16", 96),
    # token-major, 5 batch elements in chunks of 2, 2 and 1 (dx kernel), no ff block
    W_("bwd_host_uneven", (5, 77, 192), 2, 1, 192, 0, 3, 64, A.ACT_NONE, 0.0, True, "bf16", 97),
    # grouped-query heads with partial rotary: the gradients' k/v chunks follow the groups
    W_("bwd_host_gqa", (2, 200, 256), 2, 1, 256, 0, 8, 32, A.ACT_NONE, 10000.0, True, "bf16", 99,
       rope_n_elem=16, n_query_groups=2),
]


@pytest.mark.parametrize("w", BWD_CASES, ids=lambda w: w.name)
def test_backward_host_matches_oracle_and_device_path(w, cuda_ok):
    """dx, dW and db of the host entry point against the oracle; dx bit for bit
    against fp_backward (each chunk computes its rows exactly as the whole call
    does); dW and db, summed over the chunks in another order, within the f32
    rule of fp_backward's."""
    inp = fpsynth.make_inputs(w)
    grads = fpsynth.make_grads(w)
    ref = oracle.backward_workload(w, inp, grads)
    proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base,
                               w.n_query_groups, w.rope_n_elem, w.k_transposed)
    W = to_device(inp["W"], w.dtype)
    b = to_device(inp["b"], w.dtype)
    hg = tuple(None if grads[k] is None else pinned(grads[k], w.dtype)
               for k in ("ff", "q", "k", "v"))
    dx, dW, db = proj.backward_host(pinned(inp["x"], w.dtype), W, b, hg,
                                    channel_dim=w.channel_dim, n_batch_dims=w.n_batch_dims)
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_OK
    assert dx.device.type == "cpu" and dW.device.type == "cpu"
    ddx, ddW, ddb = proj.backward(to_device(inp["x"], w.dtype), W, b,
                                  tuple(None if g is None else g.cuda() for g in hg),
                                  channel_dim=w.channel_dim, n_batch_dims=w.n_batch_dims)
    torch.cuda.synchronize()
    assert torch.equal(dx, ddx.cpu()), "dx differs from fp_backward"
    perm = [a for a in range(dx.dim()) if a != w.channel_dim] + [w.channel_dim]
    assert_close(host(dx.permute(*perm).reshape(-1, w.C)), ref["dx"], "bf16", f"{w.name}:dx")
    assert_close(dW.double().numpy(), ref["dW"], "bf16", f"{w.name}:dW")
    assert_close(dW.double().numpy(), ddW.double().cpu().numpy(), "f32", f"{w.name}:dW vs device")
    assert_close(db.double().numpy(), ref["db"], "f32", f"{w.name}:db")
    assert_close(db.double().numpy(), ddb.double().cpu().numpy(), "f32", f"{w.name}:db vs device")


def test_backward_host_rejects(cuda_ok):
    """A strided x (dx would overwrite its gaps) and pageable gradients."""
    w = BWD_CASES[0]
    inp = fpsynth.make_inputs(w)
    grads = fpsynth.make_grads(w)
    proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base)
    W = to_device(inp["W"], w.dtype)
    b = to_device(inp["b"], w.dtype)
    hg = [pinned(grads[k], w.dtype) for k in ("ff", "q", "k", "v")]
    x = pinned(inp["x"], w.dtype)
    dx = torch.empty_like(x).pin_memory()
    dW = torch.empty((w.C, w.N), dtype=torch.float32).pin_memory()
    db = torch.empty((w.N,), dtype=torch.float32).pin_memory()
    big = torch.zeros((2, 4, 64, 16, 16, 1), dtype=x.dtype).pin_memory()
    big[:, :3] = x
    xs = big[:, :3]
    Ls = fpx.make_layout(xs.shape, xs.stride(), w.channel_dim, w.n_batch_dims, fpx.FP_BF16)
    call = lambda xt, L, gs: fpx.fp_backward_host(
        proj.plan, xt.data_ptr(), L, W.data_ptr(), b.data_ptr(), None,
        *[g.data_ptr() for g in gs], dx.data_ptr(), dW.data_ptr(), db.data_ptr(), None)
    assert call(xs, Ls, hg) == fpx.FP_ERR_UNSUPPORTED_LAYOUT
    L = fpx.make_layout(x.shape, x.stride(), w.channel_dim, w.n_batch_dims, fpx.FP_BF16)
    pageable = [hg[0].clone()] + hg[1:]  # clone() of a pinned tensor is pageable
    assert not pageable[0].is_pinned()
    assert call(x, L, pageable) == fpx.FP_ERR_INVALID_ARG
    assert "page-locked" in fpx.fp_last_error()
