"""GPU parity of the backward (fp_backward) against the oracle.

Small cases compare every element of dx, dW and db; the benchmark-size
workloads compare sampled token rows of dx and sampled fused columns of dW and
db (the oracle evaluates those one by one). Tolerances: the upstream gradient
path rounds G to bf16 before the two GEMMs, so dx and dW take the bf16 rule of
the forward; db is summed from the fp32 G and takes the f32 rule.
"""
import numpy as np
import pytest
import torch

import ff_input_projection_gb300 as fpx
import fpsynth
import oracle
from tests.gpu_util import assert_close, host, to_device

pytestmark = pytest.mark.gpu

W_ = fpsynth.Workload
A = fpsynth

SMALL = [
    # channels-first x: dx^T = W G^T kernel, dW with tokens contiguous
    W_("bwd_walrus_small", (2, 3, 64, 16, 16, 1), 2, 1, 64, 128, 2, 32, A.ACT_GELU_ERF, 10000.0,
       True, "bf16", 61),
    W_("bwd_walrus_ragged", (2, 3, 64, 10, 20, 1), 2, 1, 64, 128, 2, 32, A.ACT_GELU_ERF, 10000.0,
       True, "bf16", 62),
    W_("bwd_unet", (2, 96, 24, 24), 1, 1, 96, 0, 3, 32, A.ACT_NONE, 0.0, False, "bf16", 63),
    # token-major x: dx = G W^T kernel, dW with channels contiguous
    W_("bwd_bert_ff", (4, 100, 128), 2, 1, 128, 512, 0, 0, A.ACT_GELU_ERF, 0.0, True, "bf16", 64),
    W_("bwd_bert_qkv", (3, 77, 192), 2, 1, 192, 0, 3, 64, A.ACT_NONE, 0.0, True, "bf16", 65),
    W_("bwd_llm_rope", (2, 300, 256), 2, 1, 256, 0, 2, 128, A.ACT_NONE, 10000.0, False, "bf16",
       66),
    W_("bwd_rope_hd96", (2, 130, 192), 2, 1, 192, 0, 2, 96, A.ACT_NONE, 10000.0, True, "bf16", 67),
    W_("bwd_silu", (2, 3, 64, 8, 8, 1), 2, 1, 64, 192, 2, 32, A.ACT_SILU, 500.0, True, "bf16", 68),
    W_("bwd_gelu_tanh", (3, 200, 96), 2, 1, 96, 64, 0, 0, A.ACT_GELU_TANH, 0.0, True, "bf16", 69),
    W_("bwd_relu2", (2, 3, 64, 8, 16, 1), 2, 1, 64, 192, 2, 32, A.ACT_RELU2, 0.0, True, "bf16", 70),
    W_("bwd_c48_ragged", (2, 70, 48), 2, 1, 48, 48, 1, 48, A.ACT_GELU_ERF, 0.0, True, "bf16", 71),
    W_("bwd_gqa_partial", (2, 200, 256), 2, 1, 256, 0, 8, 32, A.ACT_NONE, 10000.0, True, "bf16",
       72, rope_n_elem=16, n_query_groups=2),
    W_("bwd_k_transposed", (2, 3, 64, 8, 16, 1), 2, 1, 64, 64, 2, 32, A.ACT_GELU_ERF, 10000.0,
       True, "bf16", 73, k_transposed=True),
    # rotated half-width 2: the lane-by-lane gather
    W_("bwd_rope_n4", (2, 90, 64), 2, 1, 64, 0, 2, 32, A.ACT_NONE, 10000.0, True, "bf16", 74,
       rope_n_elem=4),
    # head_dim 16, fully rotated: one rotation-pair item per head
    W_("bwd_hd16_rope", (2, 150, 64), 2, 1, 64, 0, 4, 16, A.ACT_NONE, 10000.0, True, "bf16", 75),
    # channels-first, three 128-channel row tiles: the dx^T GEMM on CTA pairs
    # with a phantom tile in the second pair, ragged token tiles
    W_("bwd_cf_c384", (2, 384, 10, 16, 1), 1, 1, 384, 128, 6, 64, A.ACT_SILU, 10000.0, True,
       "bf16", 76),
    # sequences shorter than a gather block's tokens: positions wrap several
    # times inside one block (16-byte gather, then the lane-by-lane one)
    W_("bwd_short_seq", (7, 20, 128), 2, 1, 128, 0, 2, 64, A.ACT_NONE, 10000.0, True, "bf16", 79),
    W_("bwd_short_seq_n4", (9, 11, 64), 2, 1, 64, 64, 2, 32, A.ACT_GELU_ERF, 500.0, True, "bf16",
       80, rope_n_elem=4),
]


def _proj(w):
    return fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base,
                               w.n_query_groups, w.rope_n_elem, w.k_transposed)


def run_backward(w, inp, grads, proj=None, pos=None):
    proj = proj or _proj(w)
    x = to_device(inp["x"], w.dtype)
    W = to_device(inp["W"], w.dtype)
    b = to_device(inp["b"], w.dtype)
    g = tuple(to_device(grads[k], w.dtype) for k in ("ff", "q", "k", "v"))
    pos_t = None if pos is None else torch.from_numpy(np.asarray(pos, np.int32)).cuda()
    dx, dW, db = proj.backward(x, W, b, g, pos_t, channel_dim=w.channel_dim,
                               n_batch_dims=w.n_batch_dims)
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_OK, fpx.fp_last_error()
    # dx in token order [M, C]
    nd = dx.dim()
    perm = [a for a in range(nd) if a != w.channel_dim] + [w.channel_dim]
    dx_tok = dx.permute(*perm).reshape(-1, w.C)
    return host(dx_tok), dW.double().cpu().numpy(), \
        (None if db is None else db.double().cpu().numpy())


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_backward_small(w, cuda_ok):
    inp = fpsynth.make_inputs(w)
    grads = fpsynth.make_grads(w)
    pos = None
    if w.rope_base > 0:
        pos = (np.arange(w.T, dtype=np.int32) * 7 + 2) % 1009
        inp = {**inp, "pos": pos}
    dx, dW, db = run_backward(w, inp, grads, pos=pos)
    ref = oracle.backward_workload(w, inp, grads)
    assert_close(dx, ref["dx"], "bf16", f"{w.name}:dx")
    assert_close(dW, ref["dW"], "bf16", f"{w.name}:dW")
    if w.bias:
        assert_close(db, ref["db"], "f32", f"{w.name}:db")


FULL = ["walrus_bf16", "bert_ff_bf16", "bert_qkv_bf16", "llm_qkv_rope_bf16", "unet_qkv_bf16",
        "gqa_rope_toy_bf16"]


@pytest.mark.parametrize("name", FULL)
def test_backward_full_size_sampled(name, cuda_ok):
    w = fpsynth.WORKLOADS[name]
    inp = fpsynth.make_inputs(w)
    grads = fpsynth.make_grads(w)
    dx, dW, db = run_backward(w, inp, grads)
    rng = np.random.default_rng(5)
    rows = sorted(set([0, w.M - 1] + rng.integers(0, w.M, 14).tolist()))
    cols = sorted(c for c in set([0, w.N - 1, w.F, max(w.F - 1, 0)] +
                                 rng.integers(0, w.N, 12).tolist()) if c < w.N)
    r = oracle.backward_workload(w, inp, grads, rows=rows)
    c = oracle.backward_workload(w, inp, grads, cols=cols)
    # rms floors from the whole sampled reference block
    assert_close(dx[rows], r["dx"], "bf16", f"{name}:dx-rows")
    assert_close(dW[:, cols], c["dW"], "bf16", f"{name}:dW-cols")
    if w.bias:
        assert_close(db[cols], c["db"], "f32", f"{name}:db-cols",
                     rms=float(np.sqrt(np.mean(c["db"] ** 2))))


def test_backward_rejects_f32(cuda_ok):
    w = A.WORKLOADS["tiny_fp32"]
    inp = fpsynth.make_inputs(w)
    grads = fpsynth.make_grads(w)
    proj = _proj(w)
    x = to_device(inp["x"], "f32")
    with pytest.raises(TypeError):
        proj.backward(x, to_device(inp["W"], "f32"), None,
                      tuple(to_device(grads[k], "f32") for k in ("ff", "q", "k", "v")),
                      channel_dim=w.channel_dim)


@pytest.mark.parametrize("max_ctas,cluster", [(40, 2), (152, 1), (7, 2)],
                         ids=["ctas40", "single_cta", "ctas7"])
def test_backward_launch_shapes(max_ctas, cluster, cuda_ok):
    """Other launch shapes than the default grid: with fewer than 52 CTAs the
    gather runs before the ff gradient on one stream instead of beside it; with
    the cluster option at 1 the dx and dW GEMMs run on single CTAs; an odd CTA
    cap rounds the pair grids down to whole clusters."""
    w = W_("bwd_shapes", (2, 3, 64, 16, 16, 1), 2, 1, 64, 128, 2, 32, A.ACT_GELU_ERF, 10000.0,
           True, "bf16", 77)
    inp = fpsynth.make_inputs(w)
    grads = fpsynth.make_grads(w)
    pos = (np.arange(w.T, dtype=np.int32) * 5 + 1) % 997
    inp = {**inp, "pos": pos}
    proj = _proj(w)
    proj.set_option(fpx.FP_OPT_MAX_CTAS, max_ctas)
    proj.set_option(fpx.FP_OPT_CLUSTER, cluster)
    dx, dW, db = run_backward(w, inp, grads, proj=proj, pos=pos)
    ref = oracle.backward_workload(w, inp, grads)
    assert_close(dx, ref["dx"], "bf16", "dx")
    assert_close(dW, ref["dW"], "bf16", "dW")
    assert_close(db, ref["db"], "f32", "db")


def test_backward_empty_input_zeroes_dw_db(cuda_ok):
    """No tokens: dx is empty, dW and db come back zero (they are overwritten)."""
    w = W_("bwd_empty", (0, 64, 8, 8), 1, 1, 64, 64, 4, 16, A.ACT_GELU_ERF, 0.0, True, "bf16", 78)
    proj = _proj(w)
    x = torch.empty((0, 64, 8, 8), dtype=torch.bfloat16, device="cuda")
    W = torch.randn((64, proj.N), device="cuda").to(torch.bfloat16)
    b = torch.randn((proj.N,), device="cuda").to(torch.bfloat16)
    g = (torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"),) + tuple(
        torch.empty((0, 64, 16), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    dx, dW, db = proj.backward(x, W, b, g, channel_dim=1)
    torch.cuda.synchronize()
    assert dx.numel() == 0
    assert torch.count_nonzero(dW).item() == 0 and torch.count_nonzero(db).item() == 0
    assert proj.last_launch_count == 0
