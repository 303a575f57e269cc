"""GPU path vs the CPU oracle, through the C ABI (needs a GB300).

Small shapes and the full-size workloads compare every output element;
properties that hold at any size are checked at the largest shape. Tolerances: bf16 |d| <= max(1e-2 |ref|, 2e-2 rms(ref)),
f32 |d| <= max(1e-4 |ref|, 2e-4 rms(ref)); layout/scatter with an identity
weight is bit-exact.
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

# Small cases: several tiles in M and N plus ragged tails, every path of the epilogue.
SMALL = [
    A.WORKLOADS["tiny_fp32"],
    W_("walrus_small", (2, 3, 64, 16, 16, 1), 2, 1, 64, 128, 2, 32, A.ACT_GELU_ERF, 10000.0, True,
       "bf16", 21),
    W_("walrus_ragged", (2, 3, 64, 10, 20, 1), 2, 1, 64, 128, 2, 32, A.ACT_GELU_ERF, 10000.0, True,
       "bf16", 22),
    W_("bert_ff_small", (4, 100, 128), 2, 1, 128, 512, 0, 0, A.ACT_GELU_ERF, 0.0, True, "bf16", 23),
    W_("bert_qkv_small", (3, 77, 192), 2, 1, 192, 0, 3, 64, A.ACT_NONE, 0.0, True, "bf16", 24),
    W_("llm_rope_small", (2, 300, 256), 2, 1, 256, 0, 2, 128, A.ACT_NONE, 10000.0, False, "bf16",
       25),
    W_("unet_small", (2, 64, 24, 24), 1, 1, 64, 0, 1, 64, A.ACT_NONE, 0.0, False, "bf16", 26),
    W_("unet_small_fp32", (2, 32, 20, 20), 1, 1, 32, 0, 2, 16, A.ACT_NONE, 0.0, False, "f32", 27),
    W_("rope_hd96", (2, 130, 192), 2, 1, 192, 0, 2, 96, A.ACT_NONE, 10000.0, True, "bf16", 28),
    W_("silu_bf16", (2, 3, 64, 8, 8, 1), 2, 1, 64, 192, 2, 32, A.ACT_SILU, 500.0, True, "bf16", 29),
    W_("gelu_tanh_bf16", (3, 200, 96), 2, 1, 96, 64, 0, 0, A.ACT_GELU_TANH, 0.0, True, "bf16", 30),
    W_("fp32_rope_silu", (2, 24, 6, 10), 1, 1, 24, 36, 2, 12, A.ACT_SILU, 10000.0, True, "f32", 31),
    W_("fp32_rowmajor", (3, 50, 48), 2, 1, 48, 96, 3, 16, A.ACT_GELU_ERF, 10000.0, True, "f32", 32),
    W_("one_token", (1, 1, 64), 2, 1, 64, 64, 1, 64, A.ACT_GELU_ERF, 10000.0, True, "bf16", 33),
    # tensor-core path with sequences shorter than a tile and a warp: rows of one
    # tile span several batch elements, head stores leave the whole-head path
    W_("short_seq_tc", (7, 20, 128), 2, 1, 128, 128, 2, 64, A.ACT_GELU_ERF, 10000.0, True, "bf16",
       81),
    W_("k_tail_c48", (2, 70, 48), 2, 1, 48, 0, 1, 48, A.ACT_NONE, 0.0, True, "bf16", 34),
    # bf16 shapes the TMA path cannot describe run on the FFMA kernel
    W_("bf16_odd_spatial", (2, 64, 5, 7), 1, 1, 64, 64, 2, 32, A.ACT_GELU_ERF, 10000.0, True,
       "bf16", 40),
    W_("bf16_hd16_rope", (2, 3, 32, 8, 8, 1), 2, 1, 32, 64, 2, 16, A.ACT_GELU_TANH, 10000.0, True,
       "bf16", 41),
    # grouped-query columns + partial rotary
    A.WORKLOADS["gqa_rope_toy_bf16"],
    W_("gqa_fp32", (2, 40, 48), 2, 1, 48, 0, 4, 12, A.ACT_NONE, 10000.0, True, "f32", 43,
       rope_n_elem=8, n_query_groups=2),
    W_("gqa_bf16_full_rope", (2, 200, 256), 2, 1, 256, 0, 4, 64, A.ACT_NONE, 10000.0, True, "bf16",
       44, n_query_groups=2),
    W_("relu2_bf16", (2, 3, 64, 8, 16, 1), 2, 1, 64, 192, 2, 32, A.ACT_RELU2, 0.0, True, "bf16", 45),
    W_("relu2_fp32", (2, 40, 48), 2, 1, 48, 96, 3, 16, A.ACT_RELU2, 10000.0, True, "f32", 46),
    # k emitted pre-transposed [B*kv, hd, T]: tensor-core (full and partial rotary) and FFMA paths
    W_("kt_bf16", (2, 3, 64, 8, 16, 1), 2, 1, 64, 64, 2, 32, A.ACT_GELU_ERF, 10000.0, True, "bf16",
       47, k_transposed=True),
    W_("kt_gqa_bf16", (2, 130, 256), 2, 1, 256, 0, 8, 32, A.ACT_NONE, 10000.0, False, "bf16", 48,
       rope_n_elem=8, n_query_groups=2, k_transposed=True),
    W_("kt_fp32", (2, 24, 6, 10), 1, 1, 24, 36, 2, 12, A.ACT_SILU, 10000.0, True, "f32", 49,
       k_transposed=True),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_full_compare(w, cuda_ok):
    inp = fpsynth.make_inputs(w)
    ref = oracle.forward_workload(w, inp)
    out = run(w, inp)
    for k in ("ff", "q", "k", "v"):
        if out[k] is None:
            assert ref[k].size == 0
            continue
        assert_close(host(out[k]), ref[k], w.dtype, f"{w.name}:{k}")


def test_explicit_positions(cuda_ok):
    w = SMALL[5]
    inp = fpsynth.make_inputs(w)
    pos = ((np.arange(w.T) * 37) % 1000 + 3).astype(np.int32)
    inp["pos"] = pos
    ref = oracle.forward_workload(w, inp)
    out = run(w, inp)
    for k in ("q", "k", "v"):
        assert_close(host(out[k]), ref[k], w.dtype, f"pos:{k}")


def test_strided_views_read_in_place(cuda_ok):
    """The same logical channels-first x stored channels-last (unit channel
    stride, K-major operand) and with a padded batch stride (two outer token
    axes that cannot merge) gives the oracle's result."""
    w = SMALL[1]  # [2, 3, 64, 16, 16, 1]
    inp = fpsynth.make_inputs(w)
    ref = oracle.forward_workload(w, inp)
    x = to_device(inp["x"], w.dtype)
    cl = x.permute(0, 1, 3, 4, 5, 2).contiguous().permute(0, 1, 5, 2, 3, 4)  # channels-last storage
    assert cl.stride(2) == 1
    big = torch.zeros((2, 4, 64, 16, 16, 1), dtype=x.dtype, device="cuda")
    big[:, :3] = x
    padded = big[:, :3]  # batch stride covers 4 time slices: axes (b, t) no longer merge
    for view in (cl, padded):
        out = run(w, inp, x_dev=view)
        for k in ("ff", "q", "k", "v"):
            assert_close(host(out[k]), ref[k], w.dtype, f"view:{k}")


def test_fp32_channels_first_copy_paths(cuda_ok):
    """fp32 channels-first operands go global -> shared in 16-byte chunks when
    the channel stride, the outer token strides and N are multiples of 4
    elements, else through registers. Cases on both sides of that rule: rows of
    10 tokens at a stride of 12 (the last chunk of each row is half a chunk),
    rows at a stride of 11 (channel stride 66), and N = 90 (head_dim 10).
    Tiles without rotation or transposed k store from registers; the others
    stage the tile in shared memory. Small problems take 64-column tiles (4
    CTAs per SM), two larger ones 128-column tiles."""
    w = next(s for s in SMALL if s.name == "fp32_rope_silu")  # x [2, 24, 6, 10], N 108
    inp = fpsynth.make_inputs(w)
    ref = oracle.forward_workload(w, inp)
    x = to_device(inp["x"], w.dtype)
    W = to_device(inp["W"], w.dtype)
    b = to_device(inp["b"], w.dtype)
    for row in (12, 11):
        big = torch.zeros((2, 24, 6, row), dtype=x.dtype, device="cuda")
        big[..., :10] = x
        proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base)
        out = proj.forward(big[..., :10], W, b, None, channel_dim=w.channel_dim,
                           n_batch_dims=w.n_batch_dims)
        torch.cuda.synchronize()
        assert proj.device_status() == fpx.FP_OK
        for k, o in zip(("ff", "q", "k", "v"), out):
            assert_close(host(o), ref[k], w.dtype, f"row stride {row}:{k}")
    # N = 90; then two cases without rotation, whose tiles store straight from
    # registers: GELU ff + bias + heads over ragged token and column tiles, and
    # grouped-query heads
    for w2 in (W_("fp32_n90", (2, 20, 6, 10), 1, 1, 20, 30, 2, 10, A.ACT_SILU, 10000.0, True,
                  "f32", 78),
               W_("fp32_gelu_heads", (2, 48, 9, 15), 1, 1, 48, 96, 3, 16, A.ACT_GELU_ERF, 0.0,
                  True, "f32", 79),
               W_("fp32_gqa", (2, 64, 10, 10), 1, 1, 64, 0, 4, 16, A.ACT_NONE, 0.0, True, "f32",
                  80, n_query_groups=2),
               # on 152 SMs these two keep 128-column tiles (narrower ones would not
               # lower the largest per-SM share): register stores, then rotation
               W_("fp32_wide_tiles", (2, 320, 32, 32), 1, 1, 320, 0, 5, 64, A.ACT_NONE, 0.0,
                  True, "f32", 82),
               W_("fp32_wide_rope", (2, 128, 34, 64), 1, 1, 128, 0, 2, 64, A.ACT_NONE, 10000.0,
                  True, "f32", 83)):
        inp2 = fpsynth.make_inputs(w2)
        ref2 = oracle.forward_workload(w2, inp2)
        out2 = run(w2, inp2)
        for k in ("ff", "q", "k", "v"):
            if out2[k] is None:
                assert ref2[k].size == 0
                continue
            assert_close(host(out2[k]), ref2[k], w2.dtype, f"{w2.name}:{k}")


def test_fp32_row_major_copy_paths(cuda_ok):
    """fp32 row-major x (unit-stride channels) goes global -> shared in 16-byte
    chunks of 4 channels of one token when the token stride and N are
    multiples of 4 elements, else through registers. Cases: several row and
    column tiles with rotation, on 64- and on 128-column tiles; rows padded to
    44 with C = 42 (each token's last chunk holds 2 channels); rows padded to
    37 (register path)."""
    cases = [
        (W_("fp32_km_tiles", (4, 300, 64), 2, 1, 64, 128, 4, 16, A.ACT_SILU, 10000.0, True, "f32",
            84), None),
        # 32 row tiles: on 152 SMs 128-column tiles (96 of them) keep the per-SM share
        (W_("fp32_km_wide", (4, 1000, 64), 2, 1, 64, 128, 4, 16, A.ACT_SILU, 10000.0, True, "f32",
            87), None),
        (W_("fp32_km_c42", (2, 30, 42), 2, 1, 42, 14, 3, 14, A.ACT_GELU_ERF, 0.0, True, "f32", 85),
         44),
        (W_("fp32_km_odd_stride", (2, 30, 36), 2, 1, 36, 0, 3, 12, A.ACT_NONE, 10000.0, True,
            "f32", 86), 37),
    ]
    for w, row in cases:
        inp = fpsynth.make_inputs(w)
        ref = oracle.forward_workload(w, inp)
        view = None
        if row is not None:
            x = to_device(inp["x"], w.dtype)
            big = torch.zeros(x.shape[:-1] + (row,), dtype=x.dtype, device="cuda")
            big[..., :w.C] = x
            view = big[..., :w.C]
        out = run(w, inp, x_dev=view)
        for k in ("ff", "q", "k", "v"):
            if out[k] is None:
                assert ref[k].size == 0
                continue
            assert_close(host(out[k]), ref[k], w.dtype, f"{w.name}:{k}")


def test_identity_weight_layout_is_bit_exact(cuda_ok):
    """W = [I | I | I | I], no bias/act/rotation: ff = x and q = k = v = x split
    head-major, exactly, at the full channels-first Walrus shape."""
    shape, C, h, hd = (4, 6, 768, 32, 32, 1), 768, 12, 64
    g = torch.Generator().manual_seed(5)
    x = torch.randn(shape, generator=g).to(torch.bfloat16)
    W = torch.cat([torch.eye(C)] * 4, dim=1).to(torch.bfloat16)
    proj = fpx.FusedProjection(C, C, h, hd, "none", 0.0)
    ff, q, k, v = proj.forward(x.cuda(), W.cuda(), None, None, channel_dim=2, n_batch_dims=1)
    torch.cuda.synchronize()
    B, T = 4, 6 * 32 * 32
    X = x.permute(0, 1, 3, 4, 5, 2).reshape(B * T, C)  # tokens x channels
    assert torch.equal(ff.cpu(), X)
    Xh = X.reshape(B, T, h, hd).transpose(1, 2).flatten(end_dim=1)
    for o in (q, k, v):
        assert torch.equal(o.cpu(), Xh)


def test_identity_weight_nchw_fp32_bit_exact(cuda_ok):
    shape, C, h, hd = (2, 320, 64, 64), 320, 5, 64
    x = torch.randn(shape, generator=torch.Generator().manual_seed(6))
    W = torch.cat([torch.eye(C)] * 3, dim=1)
    proj = fpx.FusedProjection(C, 0, h, hd, "none", 0.0)
    _, q, k, v = proj.forward(x.cuda(), W.cuda(), None, None, channel_dim=1, n_batch_dims=1)
    torch.cuda.synchronize()
    Xh = x.permute(0, 2, 3, 1).reshape(2, 4096, h, hd).transpose(1, 2).flatten(end_dim=1)
    for o in (q, k, v):
        assert torch.equal(o.cpu(), Xh)


FULL = ["tiny_fp32", "walrus_bf16", "bert_ff_bf16", "bert_qkv_bf16", "llm_qkv_rope_bf16",
        "unet_qkv_bf16", "unet_qkv_fp32", "gqa_rope_toy_bf16"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_every_element(name, cuda_ok):
    """Each workload at its full size, every output element against the oracle
    (the oracle runs on all host cores). The outputs start as NaN, so an element
    the kernels never wrote fails."""
    w = fpsynth.WORKLOADS[name]
    inp = fpsynth.make_inputs(w)
    out = run(w, inp)
    ref = oracle.forward_workload(w, inp)
    for k in ("ff", "q", "k", "v"):
        if out[k] is None:
            assert ref[k].size == 0
            continue
        assert_close(host(out[k]), ref[k], w.dtype, f"{name}:{k}")


def test_full_size_rope_invariants(cuda_ok):
    """At the LLM shape: position 0 is the identity (bit-exact) and each rotated
    pair keeps its norm (within bf16 rounding)."""
    w = fpsynth.WORKLOADS["llm_qkv_rope_bf16"]
    inp = fpsynth.make_inputs(w)
    off = run(w.scaled(rope_base=0.0), inp)
    zero = run(w, inp, pos=np.zeros(w.T, np.int32))
    for k in ("q", "k", "v"):
        assert torch.equal(off[k], zero[k]), k
    on = run(w, inp)
    h = w.head_dim // 2
    for k in ("q", "k"):
        a, b = on[k].float(), off[k].float()
        na = a[..., :h] ** 2 + a[..., h:] ** 2
        nb = b[..., :h] ** 2 + b[..., h:] ** 2
        rel = ((na - nb).abs() / (nb + 1e-3)).max().item()
        assert rel < 2e-2, rel
    assert torch.equal(on["v"], off["v"])


def test_launch_count_and_status(cuda_ok):
    w = SMALL[1]
    inp = fpsynth.make_inputs(w)
    proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base)
    run(w, inp, proj=proj)
    assert proj.last_launch_count == 2  # rotary table + tensor-core GEMM
    w2 = w.scaled(rope_base=0.0)
    proj2 = fpx.FusedProjection(w2.C, w2.F, w2.heads, w2.head_dim, w2.act, w2.rope_base)
    run(w2, inp, proj=proj2)
    assert proj2.last_launch_count == 1


def test_empty_tokens_on_device(cuda_ok):
    proj = fpx.FusedProjection(64, 64, 1, 64, "gelu", 10000.0)
    x = torch.empty((0, 10, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    ff, q, k, v = proj.forward(x, W, None, None, channel_dim=2)
    assert ff.shape == (0, 64) and q.shape == (0, 10, 64)
    assert proj.last_launch_count == 0


@pytest.mark.parametrize("w", [SMALL[1], SMALL[3], SMALL[5], SMALL[8]], ids=lambda w: w.name)
def test_cluster_pairs_match_single_ctas(w, cuda_ok):
    """CTA pairs (2-SM MMAs over one weight tile, the default) and single CTAs
    give identical bits; odd M-tile counts leave one CTA of the last pair
    with nothing to store."""
    inp = fpsynth.make_inputs(w)
    outs = []
    for cl in (1, 2):
        proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base)
        proj.set_option(fpx.FP_OPT_CLUSTER, cl)
        outs.append(run(w, inp, proj=proj))
    for k in ("ff", "q", "k", "v"):
        if outs[0][k] is not None:
            assert torch.equal(outs[0][k], outs[1][k]), k
    ref = oracle.forward_workload(w, inp)
    for k in ("ff", "q", "k", "v"):
        if outs[1][k] is not None:
            assert_close(host(outs[1][k]), ref[k], w.dtype, f"{w.name}:{k}")


TABLE_CASES = [
    W_("table_bf16_full", (2, 3, 64, 8, 16, 1), 2, 1, 64, 64, 2, 32, A.ACT_GELU_ERF, 10000.0, True,
       "bf16", 71),
    W_("table_bf16_partial", (2, 130, 256), 2, 1, 256, 0, 8, 32, A.ACT_NONE, 10000.0, False, "bf16",
       72, rope_n_elem=8, n_query_groups=2),
    W_("table_fp32", (2, 24, 6, 10), 1, 1, 24, 36, 2, 12, A.ACT_SILU, 10000.0, True, "f32", 73,
       k_transposed=True),
]


@pytest.mark.parametrize("w", TABLE_CASES, ids=lambda w: w.name)
def test_caller_rope_tables(w, cuda_ok):
    """cos/sin given per lane as [T, n_rot] tables with a non-contiguous inner
    dimension (every other column of a wider buffer), filled at random like the
    rope_one_entry test."""
    inp = fpsynth.make_inputs(w)
    n = w.rope_n_elem or w.head_dim
    rng = np.random.default_rng(w.seed)
    store = (lambda a: fpsynth.f32_to_bf16_bits(a.astype(np.float32))) if w.dtype == "bf16" \
        else (lambda a: a.astype(np.float32))
    wide_c = store(rng.standard_normal((w.T, 2 * n)))
    wide_s = store(rng.standard_normal((w.T, 2 * n)))
    cos_d = to_device(wide_c, w.dtype)[:, ::2]
    sin_d = to_device(wide_s, w.dtype)[:, ::2]
    assert cos_d.stride(1) == 2
    inp["rope_cos"] = fpsynth.as_float64(np.ascontiguousarray(wide_c[:, ::2]), w.dtype)
    inp["rope_sin"] = fpsynth.as_float64(np.ascontiguousarray(wide_s[:, ::2]), w.dtype)
    ref = oracle.forward_workload(w, inp)
    proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base,
                               w.n_query_groups, w.rope_n_elem, w.k_transposed)
    x, W, b = (to_device(inp[k], w.dtype) for k in ("x", "W", "b"))
    out = proj.forward(x, W, b, None, channel_dim=w.channel_dim, rope_cos=cos_d, rope_sin=sin_d)
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_OK
    assert proj.last_launch_count == 2  # table import + GEMM
    for k, o in zip(("ff", "q", "k", "v"), out):
        if o is not None:
            assert_close(host(o), ref[k], w.dtype, f"{w.name}:{k}")
    # a later default-position call rebuilds its own table
    ref2 = oracle.forward_workload(w, {**inp, "rope_cos": None, "rope_sin": None})
    out2 = run(w, {**inp, "rope_cos": None, "rope_sin": None}, proj=proj)
    for k in ("q", "k"):
        assert_close(host(out2[k]), ref2[k], w.dtype, f"{w.name}:default:{k}")


@pytest.mark.parametrize("w", [SMALL[1], SMALL[5]], ids=lambda w: w.name)
def test_back_to_back_launches_keep_order(w, cuda_ok):
    """Launches may start their prologue while the previous kernel finishes
    (programmatic dependent launch); they must still read and write in stream
    order: a forward, a torch copy of its output, and a second forward into the
    same buffers, all enqueued without synchronising."""
    inp1 = fpsynth.make_inputs(w)
    inp2 = fpsynth.make_inputs(w, seed=w.seed + 1000)
    proj = fpx.FusedProjection(w.C, w.F, w.heads, w.head_dim, w.act, w.rope_base)
    x1, x2 = to_device(inp1["x"], w.dtype), to_device(inp2["x"], w.dtype)
    W, b = to_device(inp1["W"], w.dtype), to_device(inp1["b"], w.dtype)
    out = proj.forward(x1, W, b, None, channel_dim=w.channel_dim)
    snap = [None if o is None else o.clone() for o in out]
    out = proj.forward(x2, W, b, None, channel_dim=w.channel_dim, out=out)
    snap2 = [None if o is None else o.clone() for o in out]
    proj.forward(x1, W, b, None, channel_dim=w.channel_dim, out=out)
    torch.cuda.synchronize()
    assert proj.device_status() == fpx.FP_OK
    ref1 = oracle.forward_workload(w, inp1)
    ref2 = oracle.forward_workload(w, {**inp2, "W": inp1["W"], "b": inp1["b"]})
    for i, k in enumerate(("ff", "q", "k", "v")):
        if snap[i] is not None:
            assert_close(host(snap[i]), ref1[k], w.dtype, f"first:{k}")
            assert_close(host(snap2[i]), ref2[k], w.dtype, f"second:{k}")
            assert_close(host(out[i]), ref1[k], w.dtype, f"third:{k}")
